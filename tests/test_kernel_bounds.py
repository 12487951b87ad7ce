"""CPU checks of the numeric facts the kernels' skip tests rely on (no GPU needed).

The Gumbel-max kernel skips work for elements that cannot beat the best score found so
far. Two bounds make that exact over the whole coin grid u = (2m + 1) 2^-24,
m = 0 .. 2^23 - 1:
  - a group of elements is skipped when its largest logit / T plus 17 stays below the
    best: every noise value -ln(-ln u) is below 17;
  - an element is skipped when x / T - ln(1 - u) + 1e-3 stays below the best:
    -ln(-ln u) <= -ln(1 - u) for u in (0, 1), and 1 - u is exact on the grid.
"""
import numpy as np

GUMBEL_CAP = 17.0
MARGIN = 1e-3


def _grid():
    m = np.arange(0, 1 << 23, dtype=np.float64)
    return (2.0 * m + 1.0) * 2.0 ** -24


def test_gumbel_noise_is_below_the_group_cap():
    u = _grid()
    g = -np.log(-np.log(u))
    assert g.max() < GUMBEL_CAP
    assert abs(g.max() - 16.6355) < 1e-3  # the top of the grid, u = 1 - 2^-24


def test_cheap_bound_dominates_the_noise_on_the_grid():
    u = _grid()
    g = -np.log(-np.log(u))
    ub = -np.log(1.0 - u)
    assert (ub - g).min() >= 0.0
    # 1 - u is exact in fp32 on the grid, so the kernel's bound sees the same argument
    one_minus = (np.float32(1.0) - u.astype(np.float32)).astype(np.float64)
    np.testing.assert_array_equal(one_minus, 1.0 - u)
    # the kernel's fast log is documented to err by at most 2^-21.41 (absolute) on
    # [0.5, 2] and 3 ulp elsewhere: for these arguments (|ln| <= 16.7) under 1e-5, a
    # hundredth of the margin
    worst = max(2.0 ** -21.41, 3.0 * float(np.spacing(np.float32(ub.max()))))
    assert worst < MARGIN / 100


def test_bound_is_tight_near_one_and_loose_below():
    u = _grid()
    g = -np.log(-np.log(u))
    ub = -np.log(1.0 - u)
    assert (ub - g)[-1] < 1e-6          # u -> 1: -ln u ~ 1 - u
    assert (ub - g)[len(u) // 2] > 0.3  # u = 1/2: ln 2 against -ln ln 2
