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
    ref = [0.1234, -1.75, 2.3542, -4.1776, 5.0115]
    r = _case(ref, bf16_round(np.array(ref)))
    assert r["ok"], r


def test_bound_is_absolute_below_two():
    r = _case([1.5], [1.5 + 0.0104])
    assert not r["ok"] and r["o_max"] > 1e-2
    r = _case([1.5], [1.5 + 0.0099])
    assert r["ok"]


def test_two_to_four_is_held_to_the_stated_bound():
    # Neighbours of 2.3542 are 2.34375 (0.0104 away) and 2.359375 (0.0052):
    # its floor is 0.0052 <= 1e-2, so only the near one passes.
    r = _case([-2.3542], [-2.359375])
    assert r["ok"] and r["exempt"] == 0
    r = _case([-2.3542], [-2.34375])
    assert not r["ok"] and r["beyond_bound_gated"] == 1 and r["beyond_bound_2_4"] == 1
    # 2.0070: both neighbours (2.0 at 0.0070, 2.015625 at 0.0086) are within 1e-2.
    assert _case([2.0070], [2.0])["ok"]
    assert _case([2.0070], [2.015625])["ok"]


def test_exempt_only_where_the_floor_exceeds_the_bound():
    # 4.0115: nearest bf16 is 4.0, 0.0115 away, so no bf16 output meets 1e-2;
    # held to one ulp (2^-5) instead: either neighbour passes, nothing farther.
    r = _case([4.0115], [4.0])
    assert r["ok"] and r["exempt"] == 1 and r["beyond_bound"] == 1 and r["o_max"] == 0.0
    assert _case([4.0115], [4.03125])["ok"]
    assert not _case([4.0115], [4.0625])["ok"]
    # 4.005: floor 0.005, so the far neighbour (0.026 away) fails.
    r = _case([4.005], [4.03125])
    assert not r["ok"] and r["exempt"] == 0 and r["beyond_bound_gated"] == 1
    assert _case([4.005], [4.0])["ok"]


def test_mean_rule_follows_the_oracle_floor():
    # Every element of order one, off by 1.5e-3: the floor (~7e-4 on average)
    # is below the stated bound, so 1e-3 applies and the case fails.
    ref = np.linspace(0.3, 0.9, 64) + 1e-3 / 3
    r = _case(ref, ref + 1.5e-3, pad=0)
    assert r["floor_mean"] <= 1e-3 and r["mean_rule"] == "stated" and not r["ok"]
    # Elements of order 3-4, where the rounding floor alone averages above
    # 1e-3: no bf16 output meets the stated mean, so 2 x the floor applies.
    big = np.linspace(2.1, 3.9, 64) + 2 ** -9
    r = _case(big, bf16_round(big), pad=0)
    assert r["floor_mean"] > 1e-3 and r["mean_rule"] == "floor" and r["ok"], r
    r = _case(big, big + 3 * r["floor_mean"], pad=0)
    assert not r["ok"]


def test_lse_and_mean_bounds():
    assert not _case([0.5], [0.5], lse_delta=2e-3)["ok"]
    assert _case([0.5], [0.5], lse_delta=9e-4)["ok"]
    r = _case([0.1] * 10, [0.1 + 2e-3] * 10, pad=0)   # every element off by 2e-3
    assert not r["ok"] and r["o_mean"] > 1e-3


def test_non_finite_fails():
    assert not _case([0.5], [np.nan])["ok"]
