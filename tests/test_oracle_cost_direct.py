"""Pins of the oracle's cost model and of its direct (schedule-free)
reference, no GPU.

eq. (36) ("A Generalization of the Allreduce Operation", the algorithm with
an intermediate number of steps) is checked term by term against what the
oracle's own literal simulation of the generalized schedule counts: with unit
costs (alpha, beta, gamma) = (1, 0, 0), (0, 1, 0) and (0, 0, 1) the formula
must give the rounds, the elements each process sends and the elements each
process combines.  At P = 2^k - 1 (every N_i odd but the last, the page's
worst case, the experiments' P = 127 among them) the combines are exact and
the sends exact up to the (2^r - 1) u that the r dropped distribution steps
no longer send, which eq. (36) does not give back; at any other P the
formula is an upper bound.

``direct_f64`` is checked against the exact integer reduction on inputs
whose every float64 partial is exact, and against hand-computed values;
``normwise_rel_err`` against hand examples with known 2-norms.
"""

import math

import numpy as np
import pytest

import oracle
from oracle.chunking import ceil_log2
from oracle.cost import best_r, eq36
from oracle.direct import direct_f64, direct_int, normwise_rel_err
from oracle.elementops import Arith, f32_to_bf16_rne


def _counters(P, r, u):
    """Rounds, elements sent by each process, elements combined by each
    process, for the cyclic generalized schedule on P ranks of P*u
    elements (the oracle's literal round-by-round simulation)."""
    n = P * u
    res = oracle.run("generalized", [np.zeros(n, np.int32)] * P,
                     Arith("sum", "int32"), group="cyclic", r=r)
    sent = res.sent_per_rank()
    # the cyclic group moves every rank through every position: equal loads
    assert len(set(sent)) == 1, sent
    assert res.combines % P == 0
    return res.steps, sent[0], res.combines // P, res.info


def _unit_terms(P, m, r):
    return (eq36(P, m, 1.0, 0.0, 0.0, r),
            eq36(P, m, 0.0, 1.0, 0.0, r),
            eq36(P, m, 0.0, 0.0, 1.0, r))


@pytest.mark.parametrize("P", [3, 7, 15, 31, 63, 127])
def test_eq36_terms_equal_the_simulated_schedule_worst_case(P):
    u = 3
    m = P * u
    L = ceil_log2(P)
    for r in range(L):
        steps, sent, combined, _ = _counters(P, r, u)
        t_alpha, t_beta, t_gamma = _unit_terms(P, m, r)
        assert t_alpha == steps == 2 * L - r, (P, r)
        # eq. (36) charges the extra reduction-phase data and does not give
        # back what the r dropped distribution steps no longer send
        assert math.isclose(t_beta - (2 ** r - 1) * u, sent, rel_tol=0, abs_tol=1e-9), (P, r, t_beta, sent)
        assert math.isclose(t_gamma, combined, rel_tol=0, abs_tol=1e-9), (P, r, t_gamma, combined)


@pytest.mark.parametrize("P", [2, 4, 5, 6, 9, 12, 13, 16, 20, 33])
def test_eq36_terms_bound_the_simulated_schedule_any_P(P):
    """Where some N_i is even beyond the worst case, shared partials save
    sends and combines: the formula bounds them.  The steps stay exact, and
    at r = 0 (the bandwidth-optimal algorithm) every term is exact."""
    u = 2
    m = P * u
    L = ceil_log2(P)
    for r in range(L):
        steps, sent, combined, info = _counters(P, r, u)
        t_alpha, t_beta, t_gamma = _unit_terms(P, m, r)
        T = info["Ns"][L - r]
        assert t_alpha == steps, (P, r)
        # the dropped distribution steps would have sent (T - 1) u
        assert sent <= t_beta - (T - 1) * u + 1e-9, (P, r)
        assert combined <= t_gamma + 1e-9, (P, r)
        if r == 0:
            assert math.isclose(t_beta, sent, abs_tol=1e-9) and math.isclose(t_gamma, combined, abs_tol=1e-9)


def test_eq36_is_linear_in_the_three_costs():
    rng = np.random.default_rng(3)
    for _ in range(200):
        P = int(rng.integers(3, 129))
        m = float(rng.uniform(1, 1e9))
        r = int(rng.integers(0, ceil_log2(P)))
        a, b, g = (float(x) for x in rng.uniform(0, 10, 3))
        t = _unit_terms(P, m, r)
        assert math.isclose(eq36(P, m, a, b, g, r), a * t[0] + b * t[1] + g * t[2], rel_tol=1e-12)


def test_eq36_rejects_r_outside_its_range():
    with pytest.raises(ValueError):
        eq36(8, 100, 1, 1, 1, 3)      # r = ceil(log2 8) is the latency-optimal end, outside eq. (36)
    with pytest.raises(ValueError):
        eq36(8, 100, 1, 1, 1, -1)


def test_best_r_brute_force_on_the_simulated_costs():
    """At P = 2^k - 1 the oracle's counters price every r exactly as eq. (36)
    plus the give-back term, so the minimiser over the formula must be the
    minimiser over (alpha steps + beta (sent + give-back) + gamma combined)."""
    rng = np.random.default_rng(4)
    for P in (7, 15, 31):
        u = 2
        L = ceil_log2(P)
        cnt = [_counters(P, r, u) for r in range(L)]
        for _ in range(200):
            a, b, g = (float(10 ** x) for x in rng.uniform(-3, 1, 3))
            sim = [a * s + b * (se + (2 ** r - 1) * u) + g * c for r, (s, se, c, _i) in enumerate(cnt)]
            want = min(range(L), key=lambda r: (sim[r], r))
            got = best_r(P, P * u, a, b, g)
            assert math.isclose(sim[got], sim[want], rel_tol=1e-12)


# --- direct_f64 ---------------------------------------------------------------


@pytest.mark.parametrize("op", ["sum", "prod", "max", "min"])
def test_direct_f64_equals_the_exact_integer_reduction(op):
    """Small integers: every float64 partial is exact, so the float64
    reduction must equal the int32 one."""
    rng = np.random.default_rng(5)
    P, n = 5, 300
    ints = [rng.integers(-20, 21, n).astype(np.int32) for _ in range(P)]
    want = direct_int(ints, op).astype(np.float64)
    got = direct_f64([a.astype(np.float32) for a in ints], op, "float32")
    assert got.dtype == np.float64
    assert np.array_equal(got, want)
    # the same values held as bf16 (integers up to 256 are exact in bf16)
    got16 = direct_f64([f32_to_bf16_rne(a.astype(np.float32)) for a in ints], op, "bfloat16")
    assert np.array_equal(got16, want)


# three ranks of four elements (n != P, so a division by the wrong count shows)
_HAND = [np.array([1.0, -2.0, 0.5, 6.0], np.float32),
         np.array([3.0, 4.0, -1.5, 0.0], np.float32),
         np.array([-0.25, 8.0, 2.0, -6.0], np.float32)]


@pytest.mark.parametrize("op,want", [
    ("sum", [3.75, 10.0, 1.0, 0.0]),
    ("avg", [1.25, 10.0 / 3.0, 1.0 / 3.0, 0.0]),
    ("prod", [-0.75, -64.0, -1.5, -0.0]),
    ("max", [3.0, 8.0, 2.0, 6.0]),
    ("min", [-0.25, -2.0, -1.5, -6.0]),
])
def test_direct_f64_hand_values(op, want):
    got = direct_f64(_HAND, op, "float32")
    assert np.array_equal(got, np.array(want, np.float64)), (op, got, want)


def test_direct_f64_avg_divides_the_float64_sum_once():
    """0.1 is not exact in binary: the mean of P copies is the float64 sum
    (rounded P - 1 times, in rank order) divided once by P."""
    P = 10
    x = np.full(3, 0.1, np.float32)
    s = 0.0
    for _ in range(P):
        s = s + float(np.float32(0.1))
    got = direct_f64([x] * P, "avg", "float32")
    assert np.all(got == s / P)


def test_direct_f64_reads_bf16_bit_patterns():
    one, two, m3 = np.uint16(0x3F80), np.uint16(0x4000), np.uint16(0xC040)   # 1.0, 2.0, -3.0
    bufs = [np.array([one, m3], np.uint16), np.array([two, two], np.uint16)]
    assert np.array_equal(direct_f64(bufs, "sum", "bfloat16"), [3.0, -1.0])
    assert np.array_equal(direct_f64(bufs, "prod", "bfloat16"), [2.0, -6.0])


def test_direct_f64_rejects_unknown_ops():
    with pytest.raises(ValueError):
        direct_f64(_HAND, "xor", "float32")


# --- normwise_rel_err ---------------------------------------------------------


def test_normwise_rel_err_hand_values():
    # ||(0, 0.5)|| / ||(3, 4)|| = 0.5 / 5
    assert math.isclose(normwise_rel_err([3.0, 4.5], [3.0, 4.0]), 0.1, rel_tol=1e-15)
    # the reference is the denominator: swapping the arguments changes the value
    assert math.isclose(normwise_rel_err([3.0, 4.0], [6.0, 8.0]), 0.5, rel_tol=1e-15)
    assert math.isclose(normwise_rel_err([6.0, 8.0], [3.0, 4.0]), 1.0, rel_tol=1e-15)
    # all elements at once (a 2-D array is measured as its flattened vector)
    ref = np.array([[3.0, 0.0], [0.0, 4.0]])
    y = ref + np.array([[0.0, 0.3], [0.4, 0.0]])
    assert math.isclose(normwise_rel_err(y, ref), 0.1, rel_tol=1e-14)
    assert normwise_rel_err(ref, ref) == 0.0


def test_normwise_rel_err_is_not_the_largest_elementwise_error():
    """A tiny element with a 100% error barely moves the normwise measure."""
    e = normwise_rel_err([1.0, 2e-6], [1.0, 1e-6])
    assert math.isclose(e, 1e-6 / math.hypot(1.0, 1e-6), rel_tol=1e-12)


def test_normwise_rel_err_zero_reference():
    assert normwise_rel_err([0.0, 0.0], [0.0, -0.0]) == 0.0
    assert normwise_rel_err([0.0, 1e-30], [0.0, 0.0]) == float("inf")
