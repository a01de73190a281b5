"""Randomised agreement between the schedule compiler (C ABI, host only) and
the oracle over many (P, n, schedule, parameters): rounds, per-round
traffic, combine counts and every element's reduction tree.  The cases are
drawn by hypothesis with a fixed seed, so a failure reproduces."""

import math

import pytest

hypothesis = pytest.importorskip("hypothesis")
from hypothesis import given, settings, strategies as st  # noqa: E402

import oracle  # noqa: E402
from oracle.elementops import Symbolic, leaf_buffers, tree_str  # noqa: E402

ar = pytest.importorskip("collective_reduction_gb300")


@pytest.fixture(scope="module", autouse=True)
def lib():
    import os
    if not os.path.exists(ar.LIB_PATH):
        from collective_reduction_gb300 import build
        build.build()
    return ar.lib()


@st.composite
def schedules(draw):
    P = draw(st.integers(1, 20))
    n = draw(st.integers(1, 3 * P + 7))
    L = math.ceil(math.log2(P)) if P > 1 else 0
    Lp = (1 << (P.bit_length() - 1)).bit_length() - 1
    algo = draw(st.sampled_from(["ring", "binomial", "rd", "rh", "hybrid", "generalized", "ahc", "pipeline"]))
    kw = {}
    if algo == "hybrid":
        kw["k1"] = draw(st.integers(0, Lp))
    if algo == "generalized":
        kw["r"] = draw(st.integers(0, L))
        if P & (P - 1) == 0 and draw(st.booleans()):
            kw["group"] = "xor"
    if algo == "ahc":
        G = draw(st.integers(1, min(P, 4)))
        cuts = sorted(draw(st.lists(st.integers(1, P - 1), min_size=G - 1, max_size=G - 1, unique=True))) if P > 1 else []
        edges = [0] + cuts + [P]
        kw["group_sizes"] = [b - a for a, b in zip(edges, edges[1:])]
    if algo == "pipeline":
        kw["blocks"] = draw(st.integers(1, 6))
    phase = "allreduce"
    if algo in ("ring", "rh") or (algo == "generalized" and kw.get("r") == 0):
        phase = draw(st.sampled_from(["allreduce", "reduce_scatter", "all_gather"]))
    return P, n, algo, kw, phase


@settings(max_examples=300, deadline=None, derandomize=True)
@given(schedules())
def test_compiler_agrees_with_the_oracle(case):
    P, n, algo, kw, phase = case
    try:
        s = ar.Schedule(P, n, "float32", "max", algo, phase=phase, **kw)
    except ar.ArError as e:
        # AHC with too many chunks is the one refusal among these cases
        assert algo == "ahc" and e.name == "AR_ERR_UNSUPPORTED"
        return
    res = oracle.run(algo, leaf_buffers(P, n), Symbolic(), phase=phase, **kw)
    info = s.info()
    assert info["steps"] == res.steps
    for i in range(res.steps):
        assert s.step_sent(i) == res.sent[i]
    assert info["combines"] == res.combines
    if phase == "reduce_scatter":
        cells = [(r, e) for r, lo, hi in res.info["owner"] for e in range(lo, hi)]
    else:
        cells = [(r, e) for r in range(P) for e in range(n)]
    for r, e in cells:
        assert s.tree(r, e) == tree_str(res.bufs[r][e]), (r, e)
    s.close()
