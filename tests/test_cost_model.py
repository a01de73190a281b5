"""The step-form cost model ("A Generalization of the Allreduce Operation",
eqs. 36-37), host only: eq. (37) as the library evaluates it against a brute
force over eq. (36) written out in the oracle, the prediction against the
schedule's counters, the selection against a brute force over the same
candidates, and eq. (36)'s extra-cost terms against the compiled schedules."""

import math

import numpy as np
import pytest

from oracle.cost import best_r, eq36

ar = pytest.importorskip("collective_reduction_gb300")


@pytest.fixture(scope="module")
def lib():
    import os
    if not os.path.exists(ar.LIB_PATH):
        from collective_reduction_gb300 import build
        build.build()
    return ar.lib()


def test_eq37_picks_the_eq36_minimum(lib):
    """Per-process beta and gamma of the page are P times the engine's
    per-byte costs (the P ranks' messages share one HBM)."""
    rng = np.random.default_rng(1)
    for _ in range(3000):
        P = int(rng.integers(2, 65))
        m = int(2 ** rng.uniform(4, 32))
        alpha = float(10 ** rng.uniform(-1, 2))
        beta = float(10 ** rng.uniform(-9, -5))
        gamma = float(10 ** rng.uniform(-9, -5)) * float(rng.integers(0, 2))
        model = ar.CostModel(alpha, beta, gamma)
        want = best_r(P, m, alpha, P * beta, P * gamma)
        got = ar.optimal_r(P, m, model)
        if got != want:
            # equal costs up to rounding may tie either way
            assert math.isclose(eq36(P, m, alpha, P * beta, P * gamma, got),
                                eq36(P, m, alpha, P * beta, P * gamma, want), rel_tol=1e-12)


def test_eq37_limits(lib):
    model = ar.CostModel(5.0, 1e-7, 1e-7)
    assert ar.optimal_r(1, 1024, model) == 0
    assert ar.optimal_r(2, 1024, model) == 0
    assert ar.optimal_r(63, 16, model) == 5          # latency-bound: every step but one removed
    assert ar.optimal_r(63, 1 << 34, model) == 0     # bandwidth-bound: none removed
    rs = [ar.optimal_r(63, 1 << k, model) for k in range(4, 34)]
    assert all(a >= b for a, b in zip(rs, rs[1:]))   # more data, fewer removed steps
    assert ar.optimal_r(63, 1 << 20, ar.CostModel(5.0, 0.0, 0.0)) == 5


def test_invalid_cost_requests(lib):
    r = __import__("ctypes").c_int()
    good = ar.CostModel(1.0, 1e-7, 1e-7)
    assert lib.ar_cost_optimal_r(0, 10, good, r) == 1
    assert lib.ar_cost_optimal_r(65, 10, good, r) == 1
    assert lib.ar_cost_optimal_r(8, 0, good, r) == 1
    assert lib.ar_cost_optimal_r(8, 10, ar.CostModel(0.0, 1e-7, 1e-7), r) == 1
    assert lib.ar_cost_optimal_r(8, 10, ar.CostModel(1.0, -1.0, 1e-7), r) == 1
    assert lib.ar_cost_optimal_r(8, 10, None, r) == 1
    assert lib.ar_cost_predict(None, good, None) == 1
    assert lib.ar_cost_model_default(None) == 1
    with pytest.raises(ar.ArError):
        ar.select(65, 100, "float32", "sum")


def test_predict_is_the_counters_under_the_model(lib):
    model = ar.CostModel(3.0, 2e-7, 5e-8, 0.01)
    for algo, kw in (("ring", {}), ("binomial", {}), ("generalized", {"r": 2}), ("hybrid", {"k1": 1}),
                     ("ahc", {"group_sizes": [3, 4]}), ("pipeline", {"blocks": 4})):
        for dtype, es in (("float32", 4), ("bfloat16", 2)):
            s = ar.Schedule(7, 7000, dtype, "sum", algo, form="step", **kw)
            i = s.info()
            want = 3.0 * i["steps"] + 2e-7 * i["sent_bytes_total"] + 5e-8 * i["combines"] * es + 0.01 * i["messages"]
            assert math.isclose(ar.cost_predict(s, model), want, rel_tol=1e-12)


def _candidates(P):
    Lp = (1 << (P.bit_length() - 1)).bit_length() - 1
    L = (P - 1).bit_length()
    out = [("ring", {}), ("binomial", {}), ("rd", {}), ("rh", {})]
    out += [("hybrid", {"k1": k}) for k in range(Lp + 1)]
    out += [("generalized", {"r": r}) for r in range(L + 1)]
    return out


@pytest.mark.parametrize("P", [1, 2, 5, 8, 12, 33])
def test_select_is_the_cheapest_candidate(lib, P):
    for model in (ar.CostModel(4.0, 1.6e-7, 8e-8), ar.CostModel(50.0, 1e-9, 1e-9), ar.CostModel(0.01, 1e-6, 1e-6)):
        for n in (1, 100, 1 << 16, 1 << 24):
            costs = []
            for algo, kw in _candidates(P):
                s = ar.Schedule(P, n, "float32", "sum", algo, form="step", **kw)
                costs.append((ar.cost_predict(s, model), algo, kw))
                s.close()
            best = min(c[0] for c in costs)
            first = next(c for c in costs if c[0] == best)
            algo, params, us = ar.select(P, n, "float32", "sum", model)
            assert math.isclose(us, best, rel_tol=1e-12)
            assert algo == first[1]
            for k, v in first[2].items():
                assert params[k] == v


def test_select_regimes(lib):
    # launches dominate: a schedule with the fewest rounds (L = 6 for P = 63)
    algo, params, _us = ar.select(63, 64, "float32", "sum", ar.CostModel(100.0, 1e-12, 1e-12))
    assert ar.Schedule(63, 64, "float32", "sum", algo, **params).info()["steps"] == 6
    # bytes dominate: one of the schedules with the least traffic
    algo, params, _us = ar.select(63, 1 << 24, "float32", "sum", ar.CostModel(1e-6, 1e-6, 1e-6))
    i = ar.Schedule(63, 1 << 24, "float32", "sum", algo, **params).info()
    ring = ar.Schedule(63, 1 << 24, "float32", "sum", "ring").info()
    assert i["sent_bytes_total"] == ring["sent_bytes_total"] and i["combines"] == ring["combines"]


@pytest.mark.parametrize("P", [3, 7, 15, 31, 63])
def test_eq36_extra_terms_against_the_compiled_schedules(lib, P):
    """At P = 2^k - 1 (every N_i odd but the last: the page's worst case)
    removing r distribution steps adds exactly (2^r - 1)(2L - 2) u reduced
    bytes per process, and (2^r - 1) L u sent in the reduction phase, of which
    the r dropped distribution steps give back (2^r - 1) u: eq. (36) counts
    the former and not the latter."""
    L = math.ceil(math.log2(P))
    u = 10
    base = ar.Schedule(P, P * u, "float32", "sum", "generalized", r=0, form="step").info()
    for r in range(L):
        i = ar.Schedule(P, P * u, "float32", "sum", "generalized", r=r, form="step").info()
        assert i["combines"] - base["combines"] == P * (2 ** r - 1) * (2 * L - 2) * u
        sent = (i["sent_bytes_total"] - base["sent_bytes_total"]) // 4
        assert sent == P * ((2 ** r - 1) * L * u - (2 ** r - 1) * u)
        assert i["steps"] == 2 * L - r


def test_default_model_is_positive(lib):
    m = ar.cost_model()
    assert m.alpha_us > 0 and m.beta_us_per_byte > 0 and m.gamma_us_per_byte >= 0 and m.delta_us_per_message >= 0
    # the fitted GB300 values: a few us per round, about 3 TB/s per byte sent over all ranks
    assert 1.0 < m.alpha_us < 20.0 and 1e-7 < m.beta_us_per_byte < 1e-6


@pytest.mark.parametrize("P", [2, 3, 8, 13])
def test_message_count_closed_forms(lib, P):
    """The delta term's counter: the ring sends P messages in each of its
    2 (P - 1) rounds; RD at P = 2^k sends P in each of its log2 P rounds;
    the binomial reduce + broadcast sends P - 1 messages each way."""
    assert ar.Schedule(P, P * 100, "float32", "sum", "ring").info()["messages"] == 2 * P * (P - 1)
    assert ar.Schedule(P, P * 100, "float32", "sum", "binomial").info()["messages"] == 2 * (P - 1)
    if P & (P - 1) == 0:
        assert ar.Schedule(P, P * 100, "float32", "sum", "rd").info()["messages"] == P * (P.bit_length() - 1)
