"""CPU tests of the comparison rules in tests/parity.py (constructed cases)."""
import numpy as np

from tests.parity import bf16_round, bf16_ulp, compare


def _case(o_ref_vals, o_gpu_vals, lse_delta=0.0, pad=200):
    """One row; `pad` exactly represented elements dilute the mean so that
    the max rules can be probed on their own."""
    o_ref = np.array(list(o_ref_vals) + [0.25] * pad, dtype=np.float64).reshape(1, -1)
    o_gpu = np.array(list(o_gpu_vals) + [0.25] * pad, dtype=np.float64).reshape(1, -1)
    lse_ref = np.zeros(1)
    return compare(o_gpu, lse_ref + lse_delta, o_ref, lse_ref)


def test_bf16_helpers():
    assert bf16_round(np.array([1.0 + 2 ** -9]))[0] == 1.0      # ties to even
    assert bf16_round(np.array([1.0 + 3 * 2 ** -9]))[0] == 1.0 + 2 ** -7
    assert bf16_ulp(np.array([1.5]))[0] == 2 ** -7
    assert bf16_ulp(np.array([-2.3]))[0] == 2 ** -6
    assert bf16_ulp(np.array([4.2]))[0] == 2 ** -5


def test_exact_bf16_output_passes():
    ref = [0.1234, -1.75, 2.3542, -4.1776]
    r = _case(ref, bf16_round(np.array(ref)))
    assert r["ok"], r


def test_bound_is_absolute_below_two():
    r = _case([1.5], [1.5 + 0.0104])
    assert not r["ok"] and r["o_max"] > 1e-2
    r = _case([1.5], [1.5 + 0.0099])
    assert r["ok"]


def test_faithful_rounding_at_or_above_two():
    # |O| >= 2: one ulp (>= 0.0156) is coarser than 1e-2; either bf16
    # neighbour of the exact value is accepted, nothing farther.
    r = _case([-2.3542], [-2.34375])           # the other neighbour, |d| = 0.0104
    assert r["ok"] and r["beyond_bound"] == 1 and r["o_max"] == 0.0
    r = _case([-2.3542], [-2.3542 + 2 ** -6])  # a full ulp away
    assert not r["ok"]
    r = _case([4.1776], [4.1776 + 0.03])       # ulp = 2^-5 = 0.03125
    assert r["ok"]


def test_lse_and_mean_bounds():
    assert not _case([0.5], [0.5], lse_delta=2e-3)["ok"]
    assert _case([0.5], [0.5], lse_delta=9e-4)["ok"]
    r = _case([0.1] * 10, [0.1 + 2e-3] * 10, pad=0)   # every element off by 2e-3
    assert not r["ok"] and r["o_mean"] > 1e-3


def test_non_finite_fails():
    assert not _case([0.5], [np.nan])["ok"]
