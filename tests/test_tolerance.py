"""Pins of the parity checker itself (CPU).

Every GPU parity test ends in oracle.within_tolerance / oracle.error_report
and the gates of tests/helpers.assert_close.  A slip there (a sign, the wrong
side of a comparison, a NaN that compares as a pass, a relative error taken
over the wrong elements) would turn every parity test green without checking
anything, so each piece is held here to hand-computed values and to planted
elements just inside and just outside each bound."""
import math

import numpy as np
import pytest
import torch

import oracle

import helpers

ATOL, RTOL = 1e-2, 2e-2


# ---------------------------------------------------------------------------
# within_tolerance: |got - ref| <= atol + rtol * |ref| elementwise
# ---------------------------------------------------------------------------

def test_combined_bound_hand_values():
    ref = np.array([0.005, 1.0, -2.0, 0.0])
    got = np.array([0.0, 1.01, -2.03, 0.002])
    ok, max_abs, max_rel = oracle.within_tolerance(got, ref, ATOL, RTOL)
    assert ok
    assert max_abs == pytest.approx(0.03, abs=1e-15)
    # relative error over |ref| > 1e-2 only: 0.01 / 1 and 0.03 / 2
    assert max_rel == pytest.approx(0.015, abs=1e-15)


@pytest.mark.parametrize("ref_val", [0.0, 0.3, -0.3, 2.5, -2.5])
@pytest.mark.parametrize("sign", [1.0, -1.0])
def test_combined_bound_planted_element(ref_val, sign):
    """One element planted just inside the bound passes; just outside fails,
    on either side of the reference and for either sign of the reference."""
    ref = np.linspace(-1, 1, 64)
    ref[17] = ref_val
    bound = ATOL + RTOL * abs(ref_val)
    inside = ref.copy()
    inside[17] = ref_val + sign * bound * (1 - 1e-9)
    outside = ref.copy()
    outside[17] = ref_val + sign * bound * (1 + 1e-9)
    assert oracle.within_tolerance(inside, ref, ATOL, RTOL)[0]
    assert not oracle.within_tolerance(outside, ref, ATOL, RTOL)[0]


@pytest.mark.parametrize("bad", [math.nan, math.inf, -math.inf])
def test_combined_bound_rejects_non_finite(bad):
    ref = np.zeros(8)
    got = np.zeros(8)
    got[3] = bad
    assert not oracle.within_tolerance(got, ref, ATOL, RTOL)[0]
    # a non-finite reference never passes either
    assert not oracle.within_tolerance(ref, got, ATOL, RTOL)[0]


def test_combined_bound_empty():
    assert oracle.within_tolerance(np.zeros(0), np.zeros(0), ATOL, RTOL) == (True, 0.0, 0.0)


# ---------------------------------------------------------------------------
# error_report: max-abs and max-rel measured separately
# ---------------------------------------------------------------------------

def test_error_report_hand_values():
    ref = np.array([0.005, 0.1, -0.1, 1.0, -2.0])
    got = np.array([0.009, 0.101, -0.097, 0.99, -2.01])
    r = oracle.error_report(got, ref, rel_floor=0.1)
    assert r["nonfinite"] == 0
    assert r["max_abs"] == pytest.approx(0.01, abs=1e-15)
    # |ref| >= 0.1: errors 0.001/0.1, 0.003/0.1, 0.01/1, 0.01/2 -> 0.03 (the
    # 0.004 error at |ref| = 0.005 lies below the floor and is left out)
    assert r["max_rel"] == pytest.approx(0.03, abs=1e-12)
    assert r["rel_count"] == 4
    # the floor is inclusive: raising it past 0.1 leaves only the two large elements
    r = oracle.error_report(got, ref, rel_floor=0.1000001)
    assert r["rel_count"] == 2 and r["max_rel"] == pytest.approx(0.01, abs=1e-12)


def test_error_report_non_finite_is_infinite_error():
    ref = np.array([0.5, 0.5, 0.5])
    for bad in (math.nan, math.inf):
        got = np.array([0.5, bad, 0.5])
        r = oracle.error_report(got, ref, rel_floor=0.1)
        assert r["nonfinite"] == 1
        assert r["max_abs"] == math.inf and r["max_rel"] == math.inf
    # a NaN below the relative floor still makes max_abs infinite
    r = oracle.error_report(np.array([math.nan, 0.5]), np.array([0.0, 0.5]), rel_floor=0.1)
    assert r["max_abs"] == math.inf and r["nonfinite"] == 1


def test_error_report_sign_and_shape():
    ref = np.array([0.4, -0.4])
    assert oracle.error_report(np.array([0.41, -0.4]), ref, 0.1)["max_rel"] == pytest.approx(0.025)
    assert oracle.error_report(np.array([0.4, -0.39]), ref, 0.1)["max_rel"] == pytest.approx(0.025)
    with pytest.raises(ValueError):
        oracle.error_report(np.zeros(3), np.zeros(4), 0.1)


def test_error_report_no_element_above_floor():
    r = oracle.error_report(np.array([0.001, -0.002]), np.array([0.0, 0.0]), rel_floor=0.5)
    assert r["rel_count"] == 0 and r["max_rel"] == 0.0
    assert r["max_abs"] == pytest.approx(0.002)


# ---------------------------------------------------------------------------
# helpers.assert_close: the gates every GPU parity test applies
# ---------------------------------------------------------------------------

def _bf16_case(seed=0, n=4096):
    """Reference values in [-2, 2), where a bf16 ulp is at most 2^-6: rounding
    alone stays within the stated max-abs error of 1e-2."""
    g = torch.Generator().manual_seed(seed)
    return torch.rand(n, generator=g, dtype=torch.float64) * 4 - 2


def _as_got(values: np.ndarray, dtype: str) -> torch.Tensor:
    t = torch.from_numpy(values)
    return t.to(torch.bfloat16) if dtype == "bf16" else t.to(torch.float32)


def _exact(values: np.ndarray, dtype: str) -> np.ndarray:
    """The values as the output dtype holds them (so a planted error is exactly
    what the gates compare)."""
    return _as_got(values, dtype).double().numpy()


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_assert_close_accepts_rounded_reference(dtype):
    ref = _bf16_case().numpy()
    helpers.assert_close(_as_got(ref, dtype), ref, dtype, "rounded reference")


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_assert_close_max_abs_gate(dtype):
    """An element within the combined bound (atol + rtol |ref| > atol) but past
    the stated max-abs error must fail."""
    atol, rtol = helpers.TOL[dtype]
    ref = _exact(_bf16_case().numpy(), dtype)
    ref[5] = _exact(np.array([0.7]), dtype)[0]
    got = ref.copy()
    got[5] = _exact(np.array([ref[5] + 1.5 * atol]), dtype)[0]
    err = abs(got[5] - ref[5])
    assert atol < err <= atol + rtol * abs(ref[5]), "planted error must pass only the combined bound"
    with pytest.raises(AssertionError, match="max_abs"):
        helpers.assert_close(_as_got(got, dtype), ref, dtype, "planted abs")


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_assert_close_max_rel_gate(dtype):
    """An element above the relative floor whose error is within max-abs (and
    within the combined bound) but past the stated max-rel error must fail;
    the same relative error below the floor is left to the absolute bound."""
    atol, rtol = helpers.TOL[dtype]
    floor = helpers.REL_FLOOR[dtype]
    x = 1.2 * floor
    assert 1.5 * rtol * x < atol
    ref = _exact(np.full(256, 0.37), dtype)
    ref[9] = _exact(np.array([x]), dtype)[0]
    got = ref.copy()
    got[9] = _exact(np.array([ref[9] * (1 + 1.5 * rtol)]), dtype)[0]
    assert rtol < abs(got[9] - ref[9]) / ref[9] and abs(got[9] - ref[9]) < atol
    with pytest.raises(AssertionError, match="max_rel"):
        helpers.assert_close(_as_got(got, dtype), ref, dtype, "planted rel")
    below = ref.copy()
    below[9] = _exact(np.array([0.5 * floor]), dtype)[0]
    got_b = below.copy()
    got_b[9] = _exact(np.array([below[9] * (1 + 1.5 * rtol)]), dtype)[0]
    assert abs(got_b[9] - below[9]) < atol
    helpers.assert_close(_as_got(got_b, dtype), below, dtype, "below floor")


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_assert_close_rejects_nan(dtype):
    ref = _bf16_case().numpy()
    got = ref.copy()
    got[100] = math.nan
    with pytest.raises(AssertionError):
        helpers.assert_close(_as_got(got, dtype), ref, dtype, "planted NaN")
