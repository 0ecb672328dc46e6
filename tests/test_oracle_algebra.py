"""Pins of the oracle's scan algebra (no GPU).

Each check is independent of the oracle's own formulas: function application
for the composition, exact dyadic arithmetic, brute-force unrolled sums,
closed forms and the numbers printed by the pages.

Sources: "Mamba hardware-aware parallel associative scan"
(pwwt.cn/news/6375169) sect. 1.2, 2.1, 2.2, 3.3, 4.3, 5.1;
"Mamba (part 2): parallel scan and hardware-aware optimisation"
(scwacadex.pages.dev) sect. 2.2-2.4 and 4.3.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _apply(a, b, h):
    return a * h + b


def test_compose_is_function_application():
    # pwwt sect. 1.2 hand check: doing step 1 then step 2 equals the composed step
    rng = np.random.default_rng(1)
    for _ in range(200):
        a1, b1, a2, b2, h = rng.standard_normal(5)
        a, b = oracle.compose(a2, b2, a1, b1)
        direct = _apply(a2, b2, _apply(a1, b1, h))
        assert abs(a * h + b - direct) <= 1e-14 * (1 + abs(direct))


def test_compose_order_matters():
    # the later step stands on the left; swapping operands changes the result
    a, b = oracle.compose(2.0, 3.0, 5.0, 7.0)
    assert (a, b) == (10.0, 17.0)          # 2*(5h+7)+3 = 10h+17
    a, b = oracle.compose(5.0, 7.0, 2.0, 3.0)
    assert (a, b) == (10.0, 22.0)          # 5*(2h+3)+7 = 10h+22


def test_identity_element():
    rng = np.random.default_rng(2)
    for _ in range(100):
        a, b = rng.standard_normal(2)
        assert oracle.compose(1.0, 0.0, a, b) == (a, b)
        assert oracle.compose(a, b, 1.0, 0.0) == (a, b)


def test_associativity_dyadic_exact():
    # with a, b = k / 2^8, |k| < 2^8, every product and sum is exact in
    # double, so both bracketings must agree bit for bit (scwacadex sect. 2.3)
    rng = np.random.default_rng(3)
    for _ in range(2000):
        a1, b1, a2, b2, a3, b3 = (rng.integers(-255, 256, 6) / 256.0)
        left = oracle.compose(*oracle.compose(a3, b3, a2, b2), a1, b1)
        right = oracle.compose(a3, b3, *oracle.compose(a2, b2, a1, b1))
        assert left == right


def test_associativity_random_close():
    rng = np.random.default_rng(4)
    for _ in range(2000):
        a1, a2, a3 = rng.uniform(0, 1, 3)
        b1, b2, b3 = rng.standard_normal(3)
        la, lb = oracle.compose(*oracle.compose(a3, b3, a2, b2), a1, b1)
        ra, rb = oracle.compose(a3, b3, *oracle.compose(a2, b2, a1, b1))
        assert abs(la - ra) <= 4 * np.spacing(abs(la))
        assert abs(lb - rb) <= 8 * np.spacing(max(abs(lb), 1e-300)) + 4e-16 * (abs(b1) + abs(b2) + abs(b3))


def _brute(a, b):
    """h_t = sum_{j<=t} (prod_{j<k<=t} a_k) b_j and A_t = prod_{k<=t} a_k,
    evaluated term by term."""
    L = len(a)
    A = np.empty(L)
    B = np.empty(L)
    for t in range(L):
        A[t] = math.prod(a[: t + 1])
        s = 0.0
        for j in range(t + 1):
            s += math.prod(a[j + 1: t + 1]) * b[j]
        B[t] = s
    return A, B


@pytest.mark.parametrize("L", [1, 2, 3, 5, 8, 13, 31, 32, 33, 64])
def test_scan_orderings_agree_with_brute_force(L):
    # serial, Hillis-Steele and Blelloch (identity-padded) against the
    # unrolled closed form (pwwt sect. 2.1)
    rng = np.random.default_rng(10 + L)
    a = rng.uniform(0.2, 1.0, L)
    b = rng.standard_normal(L)
    A0, B0 = _brute(a, b)
    for fn in (oracle.scan_serial, oracle.scan_hillis_steele, oracle.scan_blelloch):
        A, B = fn(a, b)
        np.testing.assert_allclose(A, A0, rtol=1e-13, atol=0)
        np.testing.assert_allclose(B, B0, rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("L", [1, 7, 16, 64])
def test_scan_orderings_dyadic_exact(L):
    # a in {1/2, 1}, b small integers: every intermediate is exact, so all
    # orderings must agree bit for bit
    rng = np.random.default_rng(20 + L)
    a = rng.choice([0.5, 1.0], L)
    b = rng.integers(-8, 9, L).astype(np.float64)
    ref = oracle.scan_serial(a, b)
    for fn in (oracle.scan_hillis_steele, oracle.scan_blelloch):
        A, B = fn(a, b)
        assert np.array_equal(A, ref[0]) and np.array_equal(B, ref[1])


def test_geometric_series_constant_a():
    for a0 in (0.3, 0.9, 0.999):
        L = 500
        a = np.full(L, a0)
        b = np.full(L, 0.7)
        _, B = oracle.scan_serial(a, b)
        t = np.arange(1, L + 1)
        closed = 0.7 * (1 - a0 ** t) / (1 - a0)
        np.testing.assert_allclose(B, closed, rtol=1e-12)


def test_unit_a_is_prefix_sum():
    # a = 1 turns the scan into the textbook prefix sum (pwwt sect. 1.2)
    rng = np.random.default_rng(5)
    b = rng.standard_normal(300)
    A, B = oracle.scan_serial(np.ones(300), b)
    np.testing.assert_allclose(B, np.cumsum(b), rtol=1e-12, atol=1e-12)
    assert np.all(A == 1.0)
    _, B = oracle.scan_serial(np.ones(10), np.full(10, 0.25))
    np.testing.assert_array_equal(B, 0.25 * np.arange(1, 11))


@pytest.mark.parametrize("L,chunk", [(8, 4), (12, 4), (13, 4), (100, 7), (256, 256), (5, 16)])
def test_chunked_two_pass_matches_serial(L, chunk):
    # pwwt sect. 2.2/3.3 two-pass scheme, sect. 5.1 minimal repro (8, chunk 4)
    rng = np.random.default_rng(L * 31 + chunk)
    a = rng.uniform(0.5, 1.0, L)
    b = rng.standard_normal(L)
    h0 = 0.37
    A, B = oracle.scan_serial(a, b)
    href = A * h0 + B
    h, bd = oracle.scan_chunked(a, b, chunk, h0)
    np.testing.assert_allclose(h, href, rtol=1e-12, atol=1e-13)
    ends = [min((k + 1) * chunk, L) - 1 for k in range((L + chunk - 1) // chunk)]
    np.testing.assert_allclose(bd, href[ends], rtol=1e-12, atol=1e-13)


def test_chunk_boundary_states_worked_example():
    # scwacadex sect. 4.3: L = 12, chunk 4 keeps h_4, h_8, h_12, which must be
    # the serial states after steps 4, 8, 12 (1-based)
    rng = np.random.default_rng(12)
    a = rng.uniform(0.5, 1.0, 12)
    b = rng.standard_normal(12)
    _, B = oracle.scan_serial(a, b)
    _, bd = oracle.scan_chunked(a, b, 4, 0.0)
    np.testing.assert_allclose(bd, B[[3, 7, 11]], rtol=1e-13, atol=1e-14)


def test_wrong_carry_is_detected():
    # the two mistakes the page warns about (sect. 3.3 / 5.1: using the last
    # local state instead of the carried one, or the chunk's own total) give a
    # different answer on the 8-step, chunk-4 repro, so the pin has teeth
    rng = np.random.default_rng(8)
    a = rng.uniform(0.5, 0.9, 8)
    b = rng.standard_normal(8)
    _, B = oracle.scan_serial(a, b)
    Al, Bl = oracle.scan_serial(a[4:], b[4:])
    wrong = Al * 0.0 + Bl                 # second chunk started from zero
    assert np.max(np.abs(wrong - B[4:])) > 1e-3
    good = Al * B[3] + Bl                 # carried state from chunk 0
    np.testing.assert_allclose(good, B[4:], rtol=1e-13)


def test_decay_underflow_numbers_printed_by_page():
    with open(os.path.join(GOLDEN, "underflow.json")) as f:
        g = json.load(f)
    for case in g["cases"]:
        L = case["steps"]
        a = np.full(L, math.exp(case["delta_A"]))
        A, _ = oracle.scan_serial(a, np.zeros(L))
        total = A[-1]
        printed = case["printed"]
        digits = case["printed_digits"]
        # agree to the digits the page prints
        assert float(f"{total:.{digits - 1}e}") == pytest.approx(printed, rel=1e-12)
        _, bd = oracle.scan_chunked(a, np.ones(L), L, 0.0)
        assert bd.shape == (1,)


def test_softplus_pins():
    assert oracle.softplus(0.0) == pytest.approx(math.log(2.0), rel=1e-15)
    for v in (-30.0, -5.0, -0.3, 0.0, 0.7, 4.0, 40.0, 800.0):
        ref = float(np.logaddexp(0.0, v))
        assert oracle.softplus(v) == pytest.approx(ref, rel=1e-14, abs=1e-300)
        # softplus(v) - softplus(-v) = v
        assert oracle.softplus(v) - oracle.softplus(-v) == pytest.approx(v, rel=1e-13, abs=1e-13)
    for dt in (1e-3, 1e-2, 1e-1):
        inv = dt + math.log(-math.expm1(-dt))
        assert oracle.softplus(inv) == pytest.approx(dt, rel=1e-12)


def test_silu_pins():
    from scipy.special import expit
    for z in (-50.0, -3.0, -0.5, 0.0, 0.5, 3.0, 50.0):
        assert oracle.silu(z) == pytest.approx(z * float(expit(z)), rel=1e-14, abs=1e-300)
    assert oracle.silu(0.0) == 0.0
