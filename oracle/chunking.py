"""Chunk split.  TEST INFRASTRUCTURE ONLY.

"All-Reduce, in depth" (The ring algorithm, the list simulation's split
helper): a buffer of length n cut into N parts takes parts of ceil(n / N)
elements; the last parts are short or empty.  A Generalization of the
Allreduce Operation (data matrix, Fig. 3.a) assumes equal parts u = m / P and
leaves the remainder open; the ceil split is the plainest reading and is used
for every schedule, including AHC's LCM x G chunks and every sub-split.
"""


def ceil_div(a, b):
    return -(-a // b)


def split(n, N):
    """The N element ranges [lo, hi) of a length-n buffer cut into N chunks."""
    if N <= 0:
        raise ValueError("N must be positive")
    size = ceil_div(n, N) if n > 0 else 0
    out = []
    for k in range(N):
        lo = min(n, k * size)
        hi = min(n, (k + 1) * size)
        out.append((lo, hi))
    return out


def ceil_log2(P):
    """Smallest L with 2^L >= P (0 for P = 1)."""
    L = 0
    while (1 << L) < P:
        L += 1
    return L
