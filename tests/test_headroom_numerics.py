"""Numerics of producing P with headroom (CPU, no GPU).

The tensor-core kernels keep a reference maximum m per column (row) that
moves only when a score passes it by 2^4, and feed P to the MMA as the
e4m3 hi + lo parts of x = 448 p 2^-4, split through half precision.  The
attention result does not depend on m (it cancels between O and the row
sum); only the rounding of P changes.  This test bounds that rounding in the
worst case -- the tile that set m held the true maximum, so the largest x is
448 2^-4 -- against the exact softmax average, on logits N(0, sigma^2) over
the spread the configs produce (descale products 0.25 .. 4).  The bound
asked is a tenth of the bf16 output tolerance (2e-2 + 2e-2 |ref|).
"""

import numpy as np
import pytest



def _e4m3_round(x: np.ndarray) -> np.ndarray:
    """Nearest e4m3 value of x >= 0, ties to even, saturating at 448: 3
    fraction bits, so spacing 2^(e - 3) in the binade [2^e, 2^(e+1)), and
    2^-9 below 2^-6 (subnormals)."""
    a = np.asarray(x, dtype=np.float64)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    q = 2.0 ** (np.maximum(e, -6.0) - 3.0)
    return np.minimum(np.round(a / q) * q, 448.0)


def _split_hilo(x: np.ndarray, lo_shift: int) -> np.ndarray:
    """hi + lo 2^-lo_shift of x as the kernels form them: x rounded to half
    precision, hi = e4m3(x), lo = e4m3((x - hi) 2^lo_shift) (the difference is
    exact in halves)."""
    xh = x.astype(np.float16).astype(np.float64)
    hi = _e4m3_round(xh)
    lo = _e4m3_round(((xh - hi) * 2.0**lo_shift).astype(np.float16).astype(np.float64))
    return hi + lo * 2.0**-lo_shift


# (headroom, lo shift, share of the tolerance allowed): the swap-AB and
# head-grouped kernels weight their separate lo columns back (shift 4); the
# query-rows kernel accumulates hi and lo products together (no shift)
CASES = [(0, 0, 0.1), (4, 4, 0.1), (4, 0, 0.35)]


@pytest.mark.parametrize("sigma", [0.5, 1.0, 2.0, 4.0, 8.0])
@pytest.mark.parametrize("tau,lo_shift,bound", CASES)
def test_headroom_rounding_within_tolerance(sigma, tau, lo_shift, bound):
    rng = np.random.default_rng(1234 + int(sigma * 10) + tau)
    worst = 0.0
    for _ in range(8):
        z = rng.standard_normal(4096) * sigma
        v = rng.standard_normal((4096, 128))
        p = np.exp(z - z.max())
        o_ref = p @ v / p.sum()
        x = 448.0 * 2.0 ** -tau * p  # largest x = 448 2^-tau: the worst case
        o = _split_hilo(x, lo_shift) @ v / x.sum()
        worst = max(worst, float(np.max(np.abs(o - o_ref) / (2e-2 + 2e-2 * np.abs(o_ref)))))
    assert worst < bound, worst
