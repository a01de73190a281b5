"""The step-count cost model.  TEST INFRASTRUCTURE ONLY.

"A Generalization of the Allreduce Operation", the algorithm with an
intermediate number of steps: removing r distribution steps costs
(2^r - 1) ceil(log P) u extra bytes sent and, in the worst case,
(2^r - 1)(2 ceil(log P) - 2) u extra bytes reduced (u = m / P), on top of the
bandwidth-optimal algorithm's 2 ceil(log P) steps, 2 (P - 1)/P m bytes sent
and (P - 1)/P m bytes reduced; each step costs alpha, each byte sent beta and
each byte reduced gamma.  That is eq. (36), written out below for
0 <= r < ceil(log P); the page minimises it over r (eq. 37) to pick the step
count.  ``best_r`` finds the integer minimiser by trying every r.
"""

import math


def eq36(P, m, alpha, beta, gamma, r):
    """Time of the generalized allreduce with r removed distribution steps,
    P processes of m bytes, per-process costs alpha, beta, gamma."""
    L = math.ceil(math.log2(P)) if P > 1 else 0
    if not 0 <= r < max(L, 1):
        raise ValueError("eq. (36) holds for 0 <= r < ceil(log2 P)")
    u = m / P
    base = 2 * L * alpha + 2 * (P - 1) / P * m * beta + (P - 1) / P * m * gamma
    extra = (2 ** r - 1) * L * u * beta + (2 ** r - 1) * (2 * L - 2) * u * gamma
    return base - r * alpha + extra


def best_r(P, m, alpha, beta, gamma):
    """The r in 0..ceil(log2 P)-1 with the lowest eq. (36) time (the lowest r
    among equal times)."""
    L = math.ceil(math.log2(P)) if P > 1 else 0
    costs = [eq36(P, m, alpha, beta, gamma, r) for r in range(max(L, 1))]
    return min(range(len(costs)), key=lambda r: (costs[r], r))
