"""Pins of the oracle's schedules against what the pages and the mathematics
fix (no GPU): brute-force results, page-derived trees, closed-form step and
byte counts, the generalized algorithm's extra-cost statements, special cases
that reduce to textbook schedules, and the AHC example."""

import itertools

import numpy as np
import pytest

import oracle
from oracle.chunking import ceil_log2, split
from oracle.direct import direct_int
from oracle.elementops import Arith, Symbolic, leaf_buffers, tree_leaves, tree_str
from oracle.schedules import ahc_holder, ahc_layout, generalized_plan


def _pow2(P):
    return P & (P - 1) == 0


def _pow2_floor(P):
    q = 1
    while q * 2 <= P:
        q *= 2
    return q


def _cases(Ps=range(1, 17)):
    """(algo, P, params) for every schedule and parameter valid at each P."""
    for P in Ps:
        L = ceil_log2(P)
        Lp = ceil_log2(_pow2_floor(P))
        yield "ring", P, {}
        yield "binomial", P, {}
        for r in range(L + 1):
            yield "generalized", P, {"group": "cyclic", "r": r}
        yield "rd", P, {}
        yield "rh", P, {}
        for k1 in range(Lp + 1):
            yield "hybrid", P, {"k1": k1}
        if _pow2(P):
            for r in range(L + 1):
                yield "generalized", P, {"group": "xor", "r": r}
        for sizes in _partitions(P):
            yield "ahc", P, {"group_sizes": sizes}
        for m in (1, 2, 3, 5):
            yield "pipeline", P, {"blocks": m}


def _partitions(P):
    """A few contiguous groupings of P ranks for AHC."""
    out = [[P]]
    if P >= 2:
        out.append([1] * P)
        out.append([P // 2, P - P // 2])
    if P >= 5:
        out.append([2, P - 2])
    if P >= 6:
        out.append([1, 2, P - 3])
    uniq = []
    for s in out:
        if s not in uniq and min(s) >= 1:
            uniq.append(s)
    return uniq


def _expected_steps(algo, P, p):
    L = ceil_log2(P)
    Lp = ceil_log2(_pow2_floor(P))
    fold = 0 if _pow2(P) else 2   # preparation + finalization rounds
    if algo == "ring":
        return 2 * (P - 1)
    if algo == "binomial":
        return 2 * L
    if algo == "rd":
        return Lp + fold
    if algo == "rh":
        return 2 * Lp + fold
    if algo == "hybrid":
        return Lp + p["k1"] + fold
    if algo == "generalized":
        return 2 * L - p["r"]
    if algo == "ahc":
        g = p["group_sizes"]
        return 2 * (max(g) - 1) + 2 * (len(g) - 1)
    if algo == "pipeline":
        return 0 if P == 1 else 2 * (P + p["blocks"] - 2)
    raise AssertionError(algo)


@pytest.mark.parametrize("op", ["sum", "prod", "max", "min"])
def test_int32_every_schedule_equals_direct_reduction(op):
    rng = np.random.default_rng(11)
    for algo, P, p in _cases():
        for n in sorted({0, 1, P - 1, P, P + 1, 2 * P + 3, 40}):
            if n < 0:
                continue
            bufs = [rng.integers(-1000, 1001, n).astype(np.int32) for _ in range(P)]
            if op == "prod":
                bufs = [rng.integers(-3, 4, n).astype(np.int32) for _ in range(P)]
            res = oracle.run(algo, bufs, Arith(op, "int32"), **p)
            want = direct_int(bufs, op)
            for r in range(P):
                assert np.array_equal(res.bufs[r], want), (algo, P, p, n, r)
            assert res.steps == _expected_steps(algo, P, p), (algo, P, p)


def test_int32_sum_exhaustive_lengths_small_P():
    rng = np.random.default_rng(12)
    for algo, P, p in _cases(range(1, 9)):
        for n in range(0, 41):
            bufs = [rng.integers(-1000, 1001, n).astype(np.int32) for _ in range(P)]
            res = oracle.run(algo, bufs, Arith("sum", "int32"), **p)
            want = direct_int(bufs, "sum")
            assert all(np.array_equal(b, want) for b in res.bufs), (algo, P, p, n)


def test_every_rank_gets_a_complete_tree():
    """Each element of each rank is a reduction of every rank exactly once."""
    for algo, P, p in _cases():
        n = 2 * P + 1
        res = oracle.run(algo, leaf_buffers(P, n), Symbolic(), **p)
        for r in range(P):
            for e in range(n):
                assert sorted(tree_leaves(res.bufs[r][e])) == list(range(P)), (algo, P, p, r, e)


def test_ring_trees_match_page(golden):
    g = golden("ring_trees.json")
    for case in g["cases"]:
        P = case["P"]
        K = 3
        res = oracle.run("ring", leaf_buffers(P, P * K), Symbolic())
        for k, want in enumerate(case["chunk_trees"]):
            for r in range(P):
                for e in range(k * K, (k + 1) * K):
                    assert tree_str(res.bufs[r][e]) == want


def test_binomial_trees_match_page(golden):
    for case in golden("binomial_trees.json")["cases"]:
        P = case["P"]
        res = oracle.run("binomial", leaf_buffers(P, 3), Symbolic())
        for r in range(P):
            assert all(tree_str(x) == case["tree"] for x in res.bufs[r])


def test_ring_traffic_closed_forms():
    # every rank sends one chunk per round: 2(N - 1) S / N per rank when N | n
    for P in range(1, 17):
        n = 12 * P
        res = oracle.run("ring", [np.zeros(n, np.int32)] * P, Arith("sum", "int32"))
        assert res.steps == 2 * (P - 1)
        assert res.sent_per_rank() == [2 * (P - 1) * n // P] * P
        assert sum(res.sent_per_rank()) == 2 * (P - 1) * n
        assert all(s == [n // P] * P for s in res.sent)


def test_ring_ceil_split_ragged():
    assert split(1024, 3) == [(0, 342), (342, 684), (684, 1024)]
    assert split(10, 4) == [(0, 3), (3, 6), (6, 9), (9, 10)]
    assert split(2, 4) == [(0, 1), (1, 2), (2, 2), (2, 2)]
    assert split(0, 3) == [(0, 0)] * 3


def test_rd_and_rh_traffic():
    for P in (2, 4, 8, 16):
        n = 8 * P
        L = ceil_log2(P)
        z = [np.zeros(n, np.int32)] * P
        rdr = oracle.run("rd", z, Arith("sum", "int32"))
        assert rdr.sent_per_rank() == [L * n] * P            # whole vector each round
        rhr = oracle.run("rh", z, Arith("sum", "int32"))
        assert rhr.sent_per_rank() == [2 * (P - 1) * n // P] * P   # same as the ring
        halves = [s[0] for s in rhr.sent[:L]]
        assert halves == [n >> (i + 1) for i in range(L)]


def test_bandwidth_optimal_generalized_sends_like_ring():
    """Bandwidth-optimal version: same transferred data as the ring,
    2 ceil(log P) steps."""
    for P in range(1, 20):
        n = 5 * P
        res = oracle.run("generalized", [np.zeros(n, np.int32)] * P,
                         Arith("sum", "int32"), group="cyclic", r=0)
        L = ceil_log2(P)
        assert res.steps == 2 * L
        assert res.sent_per_rank() == [2 * (P - 1) * 5] * P
        assert res.combines == (P - 1) * n


def test_generalized_p7_tree_and_sends(golden):
    g = golden("generalized_p7.json")
    P, K = 7, 2
    res = oracle.run("generalized", leaf_buffers(P, P * K), Symbolic(), group="cyclic", r=0)
    want0 = g["tree_chunk0_r0"]
    for c in range(P):
        shifted = "".join(str((int(ch) + c) % P) if ch.isdigit() else ch for ch in want0)
        for r in range(P):
            for e in range(c * K, (c + 1) * K):
                assert tree_str(res.bufs[r][e]) == shifted
    for r_key, want in g["sends_per_rank_in_u"].items():
        if r_key == "comment":
            continue
        res = oracle.run("generalized", [np.zeros(P * K, np.int32)] * P,
                         Arith("sum", "int32"), group="cyclic", r=int(r_key))
        assert [s[0] // K for s in res.sent] == want
        assert all(len(set(s)) == 1 for s in res.sent)


def _reduction_counts(P, r):
    n = P
    res = oracle.run("generalized", [np.zeros(n, np.int32)] * P,
                     Arith("sum", "int32"), group="cyclic", r=r)
    L = res.info["L"]
    sends = [res.sent[i][0] for i in range(L)]
    combs = [t["combines"] for t in res.info["trace"][:L]]
    return L, sends, combs, res


def test_generalized_extra_cost_one_more_result(golden):
    """r = 1: u more data per reduction step; 2u more computation on a step
    with N_i even, u otherwise, the last step (N = 2) counting u."""
    g = golden("generalized_p7.json")
    _, _, c0, _ = _reduction_counts(7, 0)
    _, _, c1, _ = _reduction_counts(7, 1)
    assert [b - a for a, b in zip(c0, c1)] == g["extra_combines_r1_per_step"]["values"]
    for P in range(3, 70):
        L, s0, c0, res0 = _reduction_counts(P, 0)
        _, s1, c1, _ = _reduction_counts(P, 1)
        assert [b - a for a, b in zip(s0, s1)] == [1] * L, P
        Ns = res0.info["Ns"]
        want = [2 if (Ns[i] % 2 == 0 and Ns[i] > 2) else 1 for i in range(L)]
        got = [b - a for a, b in zip(c0, c1)]
        # the statement is the worst case: sharing can only save combines
        assert all(x <= y for x, y in zip(got, want)), (P, got, want)
        if P == 2 ** L - 1:
            assert got == want, P


@pytest.mark.parametrize("P", [7, 15, 31, 63, 127])
def test_generalized_extra_cost_worst_case_exact(P):
    """(2^r - 1) ceil(log P) u extra data and (2^r - 1)(2 ceil(log P) - 2) u
    extra computation, exact in the worst case (N_i even in ceil(log P) - 2
    steps, i.e. P = 2^k - 1, the experiments' P = 127 among them)."""
    L, s0, c0, _ = _reduction_counts(P, 0)
    for r in range(1, L):
        _, s, c, res = _reduction_counts(P, r)
        assert sum(s) - sum(s0) == (2 ** r - 1) * L, (P, r)
        assert sum(c) - sum(c0) == (2 ** r - 1) * (2 * L - 2), (P, r)
        assert max(t["max_live_per_position"] for t in res.info["trace"]) <= 2


def test_generalized_extra_cost_bounds_any_P():
    for P in range(3, 40):
        L, s0, c0, _ = _reduction_counts(P, 0)
        for r in range(1, L):
            _, s, c, _ = _reduction_counts(P, r)
            assert sum(s) - sum(s0) <= (2 ** r - 1) * L
            assert sum(c) - sum(c0) <= (2 ** r - 1) * (2 * L - 2)


def test_latency_optimal_sends_everything_each_step():
    for P in range(2, 20):
        L, s, _, res = _reduction_counts(P, ceil_log2(P))
        assert res.steps == L
        assert s == [P] * L


@pytest.mark.parametrize("P", [2, 4, 8, 16])
def test_xor_group_is_recursive_halving_and_doubling(P):
    """With P = 2^k and the self-inverse group the bandwidth-optimal version
    is recursive halving and the latency-optimal one recursive doubling."""
    n = 2 * P + 1
    L = ceil_log2(P)
    a = oracle.run("generalized", leaf_buffers(P, n), Symbolic(), group="xor", r=0)
    b = oracle.run("rh", leaf_buffers(P, n), Symbolic())
    assert [[tree_str(x) for x in buf] for buf in a.bufs] == \
           [[tree_str(x) for x in buf] for buf in b.bufs]
    assert a.sent == b.sent
    c = oracle.run("generalized", leaf_buffers(P, n), Symbolic(), group="xor", r=L)
    d = oracle.schedules.rd(leaf_buffers(P, n), Symbolic(), first="high")
    assert [[tree_str(x) for x in buf] for buf in c.bufs] == \
           [[tree_str(x) for x in buf] for buf in d.bufs]


@pytest.mark.parametrize("P", [1, 2, 4, 8, 16])
def test_hybrid_endpoints(P):
    L = ceil_log2(P)
    n = 3 * P + 2
    h0 = oracle.run("hybrid", leaf_buffers(P, n), Symbolic(), k1=0)
    rd_ = oracle.run("rd", leaf_buffers(P, n), Symbolic())
    assert [[tree_str(x) for x in b] for b in h0.bufs] == [[tree_str(x) for x in b] for b in rd_.bufs]
    hL = oracle.run("hybrid", leaf_buffers(P, n), Symbolic(), k1=L)
    assert hL.steps == 2 * L


def test_rd_partner_distance_order():
    res = oracle.run("rd", leaf_buffers(4, 1), Symbolic())
    assert tree_str(res.bufs[0][0]) == "((0+1)+(2+3))"
    assert tree_str(res.bufs[3][0]) == "((3+2)+(1+0))"


def test_ahc_example(golden):
    g = golden("ahc_example.json")
    sizes = g["group_sizes"]
    M, G, nch, offs = ahc_layout(sizes)
    assert (M, G, nch) == (g["lcm"], g["groups"], g["chunks"])
    holders = [tuple(ahc_holder(sizes, offs, M, gm, k) for gm in range(G)) for k in range(M)]
    segs = []
    for k, hs in enumerate(holders):
        if segs and segs[-1][1] == hs:
            segs[-1][0][1] = (k + 1) * G
        else:
            segs.append([[k * G, (k + 1) * G], hs])
    assert [s[0] for s in segs] == g["segments"]
    res = oracle.run("ahc", leaf_buffers(5, 24), Symbolic(), group_sizes=sizes)
    assert res.steps == g["steps"]


def test_ahc_special_cases_reduce_to_ring():
    """One group is the ring (its LCM x G chunks are the ring's P chunks);
    groups of one rank each make the inter-group ring over P chunks."""
    for P in range(1, 9):
        n = 3 * P + 1
        ring = oracle.run("ring", leaf_buffers(P, n), Symbolic())
        want = [[tree_str(x) for x in b] for b in ring.bufs]
        one = oracle.run("ahc", leaf_buffers(P, n), Symbolic(), group_sizes=[P])
        assert [[tree_str(x) for x in b] for b in one.bufs] == want
        singles = oracle.run("ahc", leaf_buffers(P, n), Symbolic(), group_sizes=[1] * P)
        assert [[tree_str(x) for x in b] for b in singles.bufs] == want


def test_identity_cases():
    x = [np.arange(5, dtype=np.int32)]
    for algo in ("ring", "binomial", "rd", "rh", "generalized"):
        res = oracle.run(algo, x, Arith("sum", "int32"))
        assert res.steps == 0 and np.array_equal(res.bufs[0], x[0])
    res = oracle.run("ahc", x, Arith("sum", "int32"), group_sizes=[1])
    assert res.steps == 0
    z = [np.zeros(0, np.float32)] * 6
    res = oracle.run("ring", z, Arith("sum", "float32"))
    assert all(b.size == 0 for b in res.bufs)


def test_invalid_parameters_rejected():
    z = [np.zeros(4, np.int32)] * 6
    a = Arith("sum", "int32")
    with pytest.raises(ValueError):
        oracle.run("hybrid", z, a, k1=3)      # log P' = 2 for P = 6
    with pytest.raises(ValueError):
        oracle.run("generalized", z, a, group="xor")
    with pytest.raises(ValueError):
        oracle.run("generalized", z, a, r=4)
    with pytest.raises(ValueError):
        oracle.run("ahc", z, a, group_sizes=[2, 3])
    with pytest.raises(ValueError):
        generalized_plan(12, "xor", 0)


def test_float_order_is_the_schedule_order():
    """fp32: the ring's chunk-0 value equals the chain evaluated by hand in
    the order the page fixes; other chunks equal their rotated chains."""
    rng = np.random.default_rng(3)
    P, K = 5, 7
    bufs = [rng.standard_normal(P * K).astype(np.float32) for _ in range(P)]
    res = oracle.run("ring", bufs, Arith("sum", "float32"))
    for k in range(P):
        sl = slice(k * K, (k + 1) * K)
        acc = bufs[k][sl].copy()
        for j in range(1, P):
            acc = (bufs[(k + j) % P][sl] + acc).astype(np.float32)
        for r in range(P):
            assert np.array_equal(res.bufs[r][sl], acc)


@pytest.mark.parametrize("P", [3, 5, 6, 7, 9, 12, 13, 15])
def test_non_power_of_two_fold_costs(P):
    """Reducing P to the largest power of two P' with a preparation and a
    finalization step costs 2m more data per excess process (m = its vector)
    and two more steps, which makes recursive doubling slower than the
    ceil(log P) steps of the latency-optimal generalized version."""
    n = 4 * P
    Pp = _pow2_floor(P)
    e = P - Pp
    z = [np.zeros(n, np.int32)] * P
    for algo in ("rd", "rh"):
        folded = oracle.run(algo, z, Arith("sum", "int32"))
        inner = oracle.run(algo, [np.zeros(n, np.int32)] * Pp, Arith("sum", "int32"))
        assert sum(folded.sent_per_rank()) - sum(inner.sent_per_rank()) == 2 * e * n
        assert folded.steps == inner.steps + 2
        assert folded.sent[0] == [0] * Pp + [n] * e          # excess ranks send in
        assert folded.sent[-1] == [n] * e + [0] * (P - e)    # first e ranks send back
    rd = oracle.run("rd", z, Arith("sum", "int32"))
    lat = oracle.run("generalized", z, Arith("sum", "int32"), r=ceil_log2(P))
    assert rd.steps > lat.steps == ceil_log2(P)


def test_non_power_of_two_fold_tree():
    """P = 6: rank 4 and 5 fold into ranks 0 and 1; recursive doubling on
    ranks 0..3 (distance 1, then 2); ranks 4 and 5 receive ranks 0 and 1's
    results."""
    res = oracle.run("rd", leaf_buffers(6, 1), Symbolic())
    want = {0: "(((0+4)+(1+5))+(2+3))", 1: "(((1+5)+(0+4))+(3+2))", 2: "((2+3)+((0+4)+(1+5)))",
            3: "((3+2)+((1+5)+(0+4)))"}
    for r, t in want.items():
        assert tree_str(res.bufs[r][0]) == t
    assert tree_str(res.bufs[4][0]) == want[0] and tree_str(res.bufs[5][0]) == want[1]


def test_pipeline_reduce_phase_matches_page(golden):
    """p + m - 2 parallel steps until the last unit holds every block; each
    block reaches it as the chain x_{p-1} (+) (... (+) (x_1 (+) x_0))."""
    g = golden("pipeline_reduce.json")
    for c in g["reduce_steps"]:
        p, m = c["p"], c["m"]
        n = 3 * m
        res = oracle.run("pipeline", leaf_buffers(p, n), Symbolic(), blocks=m)
        assert res.steps == 2 * c["steps"]
        # the reduce phase: rounds in which some unit sends towards p - 1
        first_half = res.sent[:c["steps"]]
        assert all(sum(s) > 0 for s in first_half)
        assert all(s[p - 1] == 0 for s in first_half)
        chain = "0"
        for i in range(1, p):
            chain = f"({i}+{chain})"
        assert all(tree_str(x) == chain for b in res.bufs for x in b)


def test_pipeline_optimal_block_count(golden):
    """The page's optimal m minimises its own runtime model."""
    for c in golden("pipeline_reduce.json")["optimal_m"]:
        n, p, tb, ts = c["n"], c["p"], c["T_byte"], c["T_start"]
        def T(m):
            return (ts + n / m * tb) * (p + m - 2)
        m_star = (n * (p - 2) * tb / ts) ** 0.5
        assert T(m_star) <= T(m_star * 0.9) and T(m_star) <= T(m_star * 1.1)
        assert T(m_star) <= min(T(m) for m in range(1, 4 * int(m_star) + 10)) * (1 + 1e-9) or m_star < 1


# --- reduce-scatter / all-gather halves ("All-Reduce, in depth", The APIs) ---

def _split_cases(Ps=range(1, 17)):
    for P in Ps:
        yield "ring", P, {}
        yield "rh", P, {}
        yield "generalized", P, {"group": "cyclic"}
        if _pow2(P):
            yield "generalized", P, {"group": "xor"}


def test_reduce_scatter_owners_are_the_pages_ranks():
    """Ring: rank r ends the reduce-scatter with chunk r + 1 (the ring
    algorithm's reduce-scatter); RH: rank r with chunk r (halving keeps the
    half whose bit matches the rank's); generalized r = 0: position 0's
    vector, whose chunk c lives on rank t_0(c) = c.  RH with P not a power of
    two: P' chunks on ranks 0..P'-1, the excess ranks own nothing."""
    for algo, P, p in _split_cases():
        n = 3 * P + 2
        res = oracle.run(algo, [np.zeros(n, np.int32)] * P, Arith("sum", "int32"), phase="reduce_scatter", **p)
        Pp = _pow2_floor(P) if algo == "rh" else P
        ch = split(n, Pp)
        want = [(((c - 1) % P) if algo == "ring" else c, *ch[c]) for c in range(Pp)]
        assert res.info["owner"] == want, (algo, P, p)


def test_reduce_scatter_leaves_owners_complete_trees(golden):
    for algo, P, p in _split_cases():
        n = 2 * P + 3
        res = oracle.run(algo, leaf_buffers(P, n), Symbolic(), phase="reduce_scatter", **p)
        owned = set()
        for rank, lo, hi in res.info["owner"]:
            for e in range(lo, hi):
                assert sorted(tree_leaves(res.bufs[rank][e])) == list(range(P)), (algo, P, p, rank, e)
                owned.add((rank, e))
        # every element has exactly one owner; nobody else is complete (P > 1)
        assert sorted(e for _r, e in owned) == list(range(n))
        if P > 1:
            for r in range(P):
                for e in range(n):
                    if (r, e) not in owned:
                        assert sorted(tree_leaves(res.bufs[r][e])) != list(range(P)), (algo, P, p, r, e)
    # the owner's tree is the page's ring tree for its chunk
    for case in golden("ring_trees.json")["cases"]:
        P, K = case["P"], 3
        res = oracle.run("ring", leaf_buffers(P, P * K), Symbolic(), phase="reduce_scatter")
        for k, want in enumerate(case["chunk_trees"]):
            for e in range(k * K, (k + 1) * K):
                assert tree_str(res.bufs[(k - 1) % P][e]) == want


@pytest.mark.parametrize("dtype", ["int32", "float32", "bfloat16"])
def test_reduce_scatter_then_all_gather_is_the_allreduce(dtype):
    """The allreduce is exactly its two halves run back to back: same values
    bit for bit, same rounds, same traffic."""
    rng = np.random.default_rng(21)
    for algo, P, p in _split_cases():
        for n in (0, 1, P - 1, 2 * P + 3, 37):
            if n < 0:
                continue
            if dtype == "int32":
                bufs = [rng.integers(-1000, 1001, n).astype(np.int32) for _ in range(P)]
            else:
                bufs = [rng.standard_normal(n).astype(np.float32) for _ in range(P)]
                if dtype == "bfloat16":
                    from oracle.elementops import f32_to_bf16_rne
                    bufs = [f32_to_bf16_rne(b) for b in bufs]
            full = oracle.run(algo, bufs, Arith("sum", dtype), **p)
            rs = oracle.run(algo, bufs, Arith("sum", dtype), phase="reduce_scatter", **p)
            ag = oracle.run(algo, rs.bufs, Arith("sum", dtype), phase="all_gather", **p)
            for r in range(P):
                assert np.array_equal(ag.bufs[r].view(np.uint8), full.bufs[r].view(np.uint8)), (algo, P, p, n, r)
            assert rs.steps + ag.steps == full.steps
            assert rs.sent + ag.sent == full.sent
            assert rs.combines == full.combines and ag.combines == 0


def test_halves_traffic_closed_forms():
    """Each half of the ring, of RH (P a power of two) and of the
    bandwidth-optimal generalized schedule moves (P - 1) n / P elements per
    rank when P divides n; the ring and generalized take P - 1 and
    ceil(log2 P) rounds per half, RH log2 P' (+ 1 for the preparation or
    finalization round otherwise)."""
    for algo, P, p in _split_cases():
        n = 8 * P
        z = [np.zeros(n, np.int32)] * P
        for phase in ("reduce_scatter", "all_gather"):
            res = oracle.run(algo, z, Arith("sum", "int32"), phase=phase, **p)
            if algo == "ring":
                assert res.steps == P - 1
            elif algo == "rh":
                assert res.steps == ceil_log2(_pow2_floor(P)) + (0 if _pow2(P) else 1)
            else:
                assert res.steps == ceil_log2(P)
            if algo != "rh" or _pow2(P):
                assert res.sent_per_rank() == [(P - 1) * n // P] * P, (algo, P, phase)


def test_all_gather_reads_only_owned_chunks():
    """Inputs outside the owned chunks never reach the result: fill them
    with a sentinel and every rank still ends with the owners' chunks."""
    rng = np.random.default_rng(22)
    for algo, P, p in _split_cases():
        n = 3 * P + 1
        owner = oracle.run(algo, [np.zeros(n, np.int32)] * P, Arith("sum", "int32"), phase="reduce_scatter",
                           **p).info["owner"]
        bufs = [np.full(n, -7777, np.int32) for _ in range(P)]
        want = np.full(n, -7777, np.int32)
        for rank, lo, hi in owner:
            v = rng.integers(0, 1000, hi - lo).astype(np.int32)
            bufs[rank][lo:hi] = v
            want[lo:hi] = v
        res = oracle.run(algo, bufs, Arith("sum", "int32"), phase="all_gather", **p)
        assert (want != -7777).all() or n == 0
        for r in range(P):
            assert np.array_equal(res.bufs[r], want), (algo, P, p, r)
        assert res.combines == 0


def test_halves_only_for_splitting_schedules():
    z = [np.zeros(8, np.int32)] * 4
    for algo, kw in (("binomial", {}), ("rd", {}), ("pipeline", {"blocks": 2}), ("generalized", {"r": 1}),
                     ("hybrid", {"k1": 1}), ("ahc", {"group_sizes": [2, 2]})):
        with pytest.raises(ValueError):
            oracle.run(algo, z, Arith("sum", "int32"), phase="reduce_scatter", **kw)
    with pytest.raises(ValueError):
        oracle.run("ring", z, Arith("sum", "int32"), phase="scatter")


# --- avg ("All-Reduce, in depth", The APIs: ncclAvg divides by N) -----------

@pytest.mark.parametrize("dtype", ["float32", "bfloat16"])
def test_avg_is_the_correctly_rounded_mean_when_sums_are_exact(dtype):
    """Small-integer inputs make every partial sum exact (|sum| <= 128 fits
    bf16's 8 significant bits), so every schedule's avg must be the mean
    sum / P rounded once to the dtype.  The expected value is taken in
    float64 and then rounded to fp32 (and on to bf16): 53 >= 2 * 24 + 2 and
    24 >= 2 * 8 + 2, so these double roundings equal one correct rounding."""
    from oracle.elementops import f32_to_bf16_rne
    rng = np.random.default_rng(31)
    for algo, P, p in _cases(range(1, 17)):
        n = 2 * P + 5
        ints = [rng.integers(-8, 9, n) for _ in range(P)]
        if dtype == "float32":
            bufs = [x.astype(np.float32) for x in ints]
        else:
            bufs = [f32_to_bf16_rne(x.astype(np.float32)) for x in ints]
        mean = (np.sum(ints, axis=0).astype(np.float64) / P).astype(np.float32)
        want = mean if dtype == "float32" else f32_to_bf16_rne(mean)
        res = oracle.run(algo, bufs, Arith("avg", dtype), **p)
        for r in range(P):
            assert np.array_equal(res.bufs[r], want), (algo, P, p, r)


def test_avg_halves():
    """A reduce-scatter's avg divides the owners' finished sums; an
    all-gather combines nothing and so divides nothing."""
    rng = np.random.default_rng(32)
    for algo, P, p in _split_cases(range(2, 13)):
        n = 3 * P + 1
        bufs = [rng.standard_normal(n).astype(np.float32) for _ in range(P)]
        rs_sum = oracle.run(algo, bufs, Arith("sum", "float32"), phase="reduce_scatter", **p)
        rs_avg = oracle.run(algo, bufs, Arith("avg", "float32"), phase="reduce_scatter", **p)
        for rank, lo, hi in rs_avg.info["owner"]:
            assert np.array_equal(rs_avg.bufs[rank][lo:hi], rs_sum.bufs[rank][lo:hi] / np.float32(P))
        ag_avg = oracle.run(algo, bufs, Arith("avg", "float32"), phase="all_gather", **p)
        ag_sum = oracle.run(algo, bufs, Arith("sum", "float32"), phase="all_gather", **p)
        for r in range(P):
            assert np.array_equal(ag_avg.bufs[r], ag_sum.bufs[r])


def test_avg_has_no_integer_form():
    with pytest.raises(ValueError):
        Arith("avg", "int32")
