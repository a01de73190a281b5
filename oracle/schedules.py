"""Literal simulations of the allreduce schedules.  TEST INFRASTRUCTURE ONLY.

Each function takes the P rank buffers (NumPy arrays, or symbolic leaf
buffers), runs the schedule round by round and returns a ``Result`` with the
final rank buffers and the counters the schedule implies: rounds, elements
sent per rank per round, and element combines.

A round is a set of simultaneous messages.  Every message payload is read from
the state before the round and then applied, as rounds of simultaneous sends
are in every page.  A message either combines into the receiver, with the
receiver's own value as the left operand, or overwrites it (copy).

Schedules and where they are defined:
  ring         "All-Reduce, in depth", The ring algorithm (reduce-scatter then
               all-gather, rank r sends to r + 1, the list simulation's chunk
               indices); also A Generalization of the Allreduce Operation,
               straightforward algorithm with a cyclic group (Fig. 5)
  binomial     "還元演算子" (Reduction operator), binomial tree: the PRAM loop
               (x_i <- x_i (+) x_{i+2^k}, i inactive once bit k is set), then
               the reverse pattern as a broadcast from p_0
  rd           Recursive Doubling: every rank combines its whole vector with
               the partner at distance 2^k, k = 0..log P - 1
  rh           Recursive Halving: reduce-scatter by halving the owned range
               with partners at distance P/2, P/4, ..., then the mirror
               all-gather
  hybrid       the classic hybrid (A Generalization of the Allreduce Operation,
               introduction and the hybrid discussion before eq. 26): k1
               halving steps, recursive doubling on the remaining block, k1
               doubling steps
  generalized  A Generalization of the Allreduce Operation, eqs. 17-44: the
               positions model over a transitive abelian group T_P (cyclic
               t_k(x) = x + k mod P, Fig. 2; or the self-inverse XOR group of
               Table 1.b for P = 2^k), r removed distribution steps
  ahc          AHC (HCCL), Description steps 1-3
  pipeline     "還元演算子" (Reduction operator), pipelined algorithm: a chain
               reduce over m blocks, then the mirror-image broadcast

The ring, rh and the generalized schedule with r = 0 split into a
reduce-scatter and an all-gather ("All-Reduce, in depth", The APIs: the two
halves are the collectives FSDP and ZeRO call on their own).  phase =
"reduce_scatter" runs the first half only, "all_gather" the second half only
on buffers whose owned chunks hold the values to spread; ``Result.info
["owner"]`` lists (rank, lo, hi): who holds the full reduction of [lo, hi)
after the first half, and so who supplies it to the second.
"""

import math

import numpy as np

from .chunking import ceil_div, ceil_log2, split

ALGOS = ("ring", "binomial", "rd", "rh", "hybrid", "generalized", "ahc", "pipeline")
PHASES = ("allreduce", "reduce_scatter", "all_gather")


def _halves(phase):
    """(run the reduce-scatter half, run the all-gather half)."""
    if phase not in PHASES:
        raise ValueError(f"unknown phase {phase!r}")
    return phase != "all_gather", phase != "reduce_scatter"


class Result:
    def __init__(self, bufs, sent, combines, info=None):
        self.bufs = bufs            # final rank buffers
        self.sent = sent            # sent[step][rank] = elements sent in that round
        self.combines = combines    # element combines performed
        self.info = info or {}

    @property
    def steps(self):
        return len(self.sent)

    def sent_per_rank(self):
        P = len(self.bufs)
        return [sum(s[r] for s in self.sent) for r in range(P)]


class RankSim:
    """P ranks, each holding one buffer; rounds of simultaneous messages."""

    def __init__(self, bufs, arith):
        self.P = len(bufs)
        self.n = len(bufs[0]) if self.P else 0
        self.arith = arith
        self.buf = [np.array(b, dtype=arith.storage, copy=True) for b in bufs]
        self.sent = []
        self.start = arith.combines

    def round(self, msgs):
        """msgs: (src, dst, lo, hi, kind), kind 'add' (combine) or 'copy'."""
        payload = [self.buf[s][lo:hi].copy() for (s, d, lo, hi, _k) in msgs]
        # a round may write each element of a destination at most once
        by_dst = {}
        for (s, d, lo, hi, _k) in msgs:
            if hi > lo:
                by_dst.setdefault(d, []).append((lo, hi))
        for d, rs in by_dst.items():
            rs.sort()
            for (a0, a1), (b0, _b1) in zip(rs, rs[1:]):
                if b0 < a1:
                    raise AssertionError(f"round writes rank {d} twice")
        sent = [0] * self.P
        for (s, d, lo, hi, kind), data in zip(msgs, payload):
            if s == d:
                raise AssertionError("a message must go to another rank")
            sent[s] += hi - lo
            if hi <= lo:
                continue
            if kind == "add":
                self.buf[d][lo:hi] = self.arith.combine(self.buf[d][lo:hi], data)
            elif kind == "copy":
                self.buf[d][lo:hi] = data
            else:
                raise ValueError(kind)
        self.sent.append(sent)

    def result(self, info=None):
        return Result(self.buf, self.sent, self.arith.combines - self.start, info)


def _is_pow2(P):
    return P >= 1 and (P & (P - 1)) == 0


def ring(bufs, arith, phase="allreduce"):
    """Ring reduce-scatter + all-gather over P chunks (ceil split).

    Reduce-scatter round t: rank r passes chunk (r - t) mod P to rank r + 1,
    which adds it into its own copy.  Afterwards rank r holds the full
    reduction of chunk (r + 1) mod P.  All-gather round t: rank r passes chunk
    (r + 1 - t) mod P to rank r + 1, which overwrites its copy.
    2(P - 1) rounds.
    """
    do_rs, do_ag = _halves(phase)
    sim = RankSim(bufs, arith)
    P, n = sim.P, sim.n
    ch = split(n, P)
    for t in range(P - 1 if do_rs else 0):
        sim.round([(r, (r + 1) % P, *ch[(r - t) % P], "add") for r in range(P)])
    for t in range(P - 1 if do_ag else 0):
        sim.round([(r, (r + 1) % P, *ch[(r + 1 - t) % P], "copy") for r in range(P)])
    return sim.result({"owner": [((c - 1) % P, *ch[c]) for c in range(P)]})


def binomial(bufs, arith):
    """Binomial-tree reduce to p_0, then broadcast from p_0.

    Reduce, k = 0..ceil(log2 P) - 1: every active unit i whose bit k is set
    sends x_i to p_{i - 2^k} and becomes inactive; every other active unit i
    with i + 2^k < P computes x_i <- x_i (+) x_{i + 2^k}.  The broadcast runs
    the same tree backwards with copies.  2 ceil(log2 P) rounds.
    """
    sim = RankSim(bufs, arith)
    P, n = sim.P, sim.n
    L = ceil_log2(P)
    active = [True] * P
    for k in range(L):
        msgs = []
        for i in range(P):
            if not active[i]:
                continue
            if (i >> k) & 1:
                active[i] = False
            elif i + (1 << k) < P:
                msgs.append((i + (1 << k), i, 0, n, "add"))
        sim.round(msgs)
    for k in reversed(range(L)):
        msgs = [(i, i + (1 << k), 0, n, "copy")
                for i in range(0, P, 1 << (k + 1)) if i + (1 << k) < P]
        sim.round(msgs)
    return sim.result()


def fold_to_pow2(bufs, arith, inner, phase="allreduce"):
    """Any P by reduction to the largest power of two P' <= P (A Generalization
    of the Allreduce Operation, introduction, the straightforward workaround
    for non-power-of-two process counts): a preparation round in which each
    excess process sends its vector to a process that takes part, the
    power-of-two schedule on the P' taking part, and a finalization round in
    which the result goes back.  Excess process P' + i pairs with process i
    (the pages leave the pairing open).  inner(bufs) runs the schedule on P'
    buffers and returns its Result.  A power-of-two P runs inner directly.
    A reduce-scatter keeps the preparation round and an all-gather the
    finalization round; the excess processes own no chunk.
    """
    do_rs, do_ag = _halves(phase)
    P = len(bufs)
    Pp = 1
    while Pp * 2 <= P:
        Pp *= 2
    if Pp == P:
        return inner(bufs)
    n = len(bufs[0])
    e = P - Pp
    pre = RankSim(bufs, arith)
    if do_rs:
        pre.round([(Pp + i, i, 0, n, "add") for i in range(e)])
    res = inner(pre.buf[:Pp])
    post = RankSim(list(res.bufs) + [pre.buf[Pp + i] for i in range(e)], arith)
    if do_ag:
        post.round([(i, Pp + i, 0, n, "copy") for i in range(e)])
    sent = pre.sent + [list(s) + [0] * e for s in res.sent] + post.sent
    # one counter serves all three parts: everything since the preparation
    combines = arith.combines - pre.start
    return Result(post.buf, sent, combines, dict(res.info, P_pow2=Pp, excess=e))


def _rd_pow2(bufs, arith, first):
    sim = RankSim(bufs, arith)
    P, n = sim.P, sim.n
    L = ceil_log2(P)
    dists = [1 << k for k in range(L)]
    if first == "high":
        dists = dists[::-1]
    for d in dists:
        sim.round([(r ^ d, r, 0, n, "add") for r in range(P)])
    return sim.result()


def rd(bufs, arith, first="low"):
    """Recursive doubling: log P rounds, x_r <- x_r (+) x_{r xor d}.

    first='low' takes distances 1, 2, 4, ... (the classic order); 'high' takes
    P/2, P/4, ..., 1.  Other P: fold_to_pow2 around it (log P' + 2 rounds).
    """
    return fold_to_pow2(bufs, arith, lambda b: _rd_pow2(b, arith, first))


def _chunk_span(ch, c0, c1):
    return ch[c0][0], ch[c1 - 1][1]


def _halving_rounds(sim, ch, own, L, steps):
    """Recursive-halving reduce-scatter rounds 0..steps-1 (distance P/2 first).

    own[r] = (c0, c1) is rank r's chunk range; each round a rank keeps the half
    holding the chunks whose bit matches its own and sends the other half to
    the partner, which combines it into the same half of its own range.
    """
    P = sim.P
    for i in range(steps):
        d = P >> (i + 1)
        msgs, nxt = [], []
        for r in range(P):
            c0, c1 = own[r]
            mid = (c0 + c1) // 2
            keep, give = ((mid, c1), (c0, mid)) if r & d else ((c0, mid), (mid, c1))
            msgs.append((r, r ^ d, *_chunk_span(ch, *give), "add"))
            nxt.append(keep)
        sim.round(msgs)
        own[:] = nxt


def _doubling_rounds(sim, ch, own, steps):
    """Mirror all-gather of ``_halving_rounds``: rounds steps-1..0, copies."""
    P = sim.P
    for i in reversed(range(steps)):
        d = P >> (i + 1)
        sim.round([(r, r ^ d, *_chunk_span(ch, *own[r]), "copy") for r in range(P)])
        own[:] = [(min(own[r][0], own[r ^ d][0]), max(own[r][1], own[r ^ d][1]))
                  for r in range(P)]


def pow2_floor(P):
    Pp = 1
    while Pp * 2 <= P:
        Pp *= 2
    return Pp


def rh(bufs, arith, phase="allreduce"):
    """Recursive halving reduce-scatter + recursive doubling all-gather.

    2 log P rounds; rank r ends the reduce-scatter with chunk r.  Other P:
    fold_to_pow2 around it (2 log P' + 2 rounds).
    """
    return hybrid(bufs, arith, ceil_log2(pow2_floor(len(bufs))), phase)


def hybrid(bufs, arith, k1, phase="allreduce"):
    """Classic hybrid: k1 halving rounds, recursive doubling (distance 1
    first) on the block each rank then owns, k1 doubling rounds.

    k1 = 0 is recursive doubling, k1 = log P is recursive halving; log P + k1
    rounds.  Other P: fold_to_pow2 around it, k1 in 0..log P'.
    """
    Lp = ceil_log2(pow2_floor(len(bufs)))
    if not 0 <= k1 <= Lp:
        raise ValueError("k1 must lie in 0..log P'")
    if phase != "allreduce" and k1 != Lp:
        raise ValueError("only recursive halving (k1 = log P') splits into halves")
    return fold_to_pow2(bufs, arith, lambda b: _hybrid_pow2(b, arith, k1, phase), phase)


def _hybrid_pow2(bufs, arith, k1, phase="allreduce"):
    do_rs, do_ag = _halves(phase)
    sim = RankSim(bufs, arith)
    P, n = sim.P, sim.n
    L = ceil_log2(P)
    ch = split(n, P)
    own = [(0, P)] * P
    if do_rs:
        _halving_rounds(sim, ch, own, L, k1)
    else:
        # the ranges the halving would leave (no messages): rank r, chunk r
        _halving_rounds(_Dry(P), ch, own, L, k1)
    owner = [(r, *_chunk_span(ch, *own[r])) for r in range(P)] if k1 == L else []
    for k in range(L - k1):
        d = 1 << k
        sim.round([(r ^ d, r, *_chunk_span(ch, *own[r]), "add") for r in range(P)])
    if do_ag:
        _doubling_rounds(sim, ch, own, k1)
    return sim.result({"owner": owner})


class _Dry:
    """Stands in for a RankSim where only the ownership bookkeeping of
    _halving_rounds is wanted: it accepts and drops every round."""

    def __init__(self, P):
        self.P = P

    def round(self, msgs):
        pass


class _Trees:
    """Interned reduction trees over vector indices (the partials q of the
    generalized algorithm): a leaf is ('v', index), a combine is (left, right)."""

    def __init__(self):
        self.ids = {}
        self.nodes = []

    def get(self, key):
        i = self.ids.get(key)
        if i is None:
            i = len(self.nodes)
            self.ids[key] = i
            self.nodes.append(key)
        return i


def generalized_plan(P, group, r):
    """The step counts of the generalized algorithm: N_0 = P,
    N_{i+1} = ceil(N_i / 2), L = ceil(log2 P) reduction steps, T = N_{L-r}
    targets, L - r distribution steps."""
    if group not in ("cyclic", "xor"):
        raise ValueError(group)
    if group == "xor" and not _is_pow2(P):
        raise ValueError("the XOR group needs a power-of-two P")
    Ns = [P]
    while Ns[-1] > 1:
        Ns.append(ceil_div(Ns[-1], 2))
    L = len(Ns) - 1
    if not 0 <= r <= L:
        raise ValueError("r must lie in 0..ceil(log2 P)")
    return Ns, L, Ns[L - r]


def generalized(bufs, arith, group="cyclic", r=0, phase="allreduce"):
    """The group-theoretic generalized allreduce.

    Positions model.  The group T_P acts on ranks: cyclic t_a(c) = (a + c)
    mod P, XOR t_a(c) = a xor c.  The distributed vector at position a holds
    chunk c on rank t_a(c); initially position a holds the data vector
    q_a (chunk c of rank t_a(c)).

    Reduction step i (N = N_i, h = floor(N / 2), lo = N - 2h): the vectors at
    positions lo+h..N-1 move by -h onto positions lo..lo+h-1 and combine
    (receiver on the left); position 0 idles when N is odd (the q*_0 of the
    bandwidth-optimal algorithm).  Removing r distribution steps requires the
    T = N_{L-r} shifted results t^s q_Sigma, s = 0..T-1: target s runs the
    same operators with every vector index shifted by s (position j of target
    s sits at absolute position s o j).  A message is one per distinct
    (absolute position, partial); a combine is one per distinct result, so
    shared partials are computed once.

    Distribution, steps i = L-r-1 down to 0: positions lo..lo+h-1 copy to +h.
    With r = L (latency-optimal) there is none, and every rank keeps its own
    target's result.

    With r = 0 the reduction steps are a reduce-scatter (position 0 ends with
    the result, so rank t_0(c) = c holds chunk c) and the distribution an
    all-gather of position 0's vector.  A reduce-scatter leaves every rank's
    other chunks as they came in; an all-gather takes position 0's vector from
    the input.
    """
    do_rs, do_ag = _halves(phase)
    P = len(bufs)
    n = len(bufs[0])
    Ns, L, T = generalized_plan(P, group, r)
    if phase != "allreduce" and r != 0:
        raise ValueError("only r = 0 splits into halves")
    ch = split(n, P)
    cyc = group == "cyclic"

    def rank_of(a, c):          # t_a(c)
        return (a + c) % P if cyc else a ^ c

    def chunk_of(a, rank):      # the chunk that rank holds of position a
        return (rank - a) % P if cyc else rank ^ a

    def comp(s, j):             # absolute position of target s, relative j
        return (s + j) % P if cyc else s ^ j

    def shift(a, h):            # the position h above a in the target frame
        return (a + h) % P if cyc else a ^ h

    def pos_of(rank, c):        # the position whose chunk c lives on rank
        return (rank - c) % P if cyc else rank ^ c

    trees = _Trees()
    values = {}
    start = arith.combines

    def vector(v):
        out = arith.empty(n)
        for c, (lo, hi) in enumerate(ch):
            out[lo:hi] = bufs[rank_of(v, c)][lo:hi]
        return out

    cur = []
    for s in range(T):
        row = []
        for j in range(P):
            a = comp(s, j)
            t = trees.get(("v", a))
            if (a, t) not in values:
                values[(a, t)] = vector(a)
            row.append(t)
        cur.append(row)

    sent, trace = [], []
    for i in range(L if do_rs else 0):
        N = Ns[i]
        h = N // 2
        lo = N - 2 * h
        msgs, combos = set(), {}
        nxt = [row[:Ns[i + 1]] for row in cur]
        for s in range(T):
            for j in range(lo, lo + h):
                a_dst, a_src = comp(s, j), comp(s, j + h)
                assert a_src == shift(a_dst, h)
                t_dst, t_src = cur[s][j], cur[s][j + h]
                msgs.add((a_src, t_src))
                t_new = trees.get((t_dst, t_src))
                combos[(a_dst, t_new)] = (t_dst, a_src, t_src)
                nxt[s][j] = t_new
        new_values = {}
        for (a_dst, t_new), (t_dst, a_src, t_src) in combos.items():
            new_values[(a_dst, t_new)] = arith.combine(values[(a_dst, t_dst)],
                                                       values[(a_src, t_src)])
        cur = nxt
        live = {}
        for s in range(T):
            for j in range(Ns[i + 1]):
                key = (comp(s, j), cur[s][j])
                live[key] = new_values[key] if key in new_values else values[key]
        values = live
        per_rank = [0] * P
        for (a_src, _t) in msgs:
            for rank in range(P):
                c = chunk_of(a_src, rank)
                per_rank[rank] += ch[c][1] - ch[c][0]
        sent.append(per_rank)
        per_pos = {}
        for (a, t) in values:
            per_pos.setdefault(a, set()).add(t)
        trace.append({"messages": len(msgs), "combines": len(combos),
                      "max_live_per_position": max(len(v) for v in per_pos.values())})

    final = {a: values[(a, cur[a][0])] for a in range(T)}
    for i in reversed(range(L - r if do_ag else 0)):
        N = Ns[i]
        h = N // 2
        lo = N - 2 * h
        per_rank = [0] * P
        for a in range(lo, lo + h):
            final[shift(a, h)] = final[a]
            for rank in range(P):
                c = chunk_of(a, rank)
                per_rank[rank] += ch[c][1] - ch[c][0]
        sent.append(per_rank)
        trace.append({"messages": h, "combines": 0, "max_live_per_position": 1})

    out = []
    for rank in range(P):
        b = arith.empty(n)
        for c, (clo, chi) in enumerate(ch):
            if pos_of(rank, c) in final:
                b[clo:chi] = final[pos_of(rank, c)][clo:chi]
            else:
                b[clo:chi] = bufs[rank][clo:chi]
        out.append(b)
    owner = [(rank_of(0, c), *ch[c]) for c in range(P)] if r == 0 else []
    info = {"L": L, "T": T, "Ns": Ns, "trace": trace, "owner": owner}
    return Result(out, sent, arith.combines - start, info)


def pipeline(bufs, arith, m):
    """Pipelined chain reduce + broadcast ("還元演算子" (Reduction operator),
    pipelined algorithm).  The vector is cut into m blocks (ceil split).
    Reduce: in round t unit i < p-1 passes block t - i (when 0 <= t - i < m)
    to unit i + 1, which combines it into its own; the last unit holds every
    block after p + m - 2 rounds (p - 1 until it receives the first block,
    m - 1 more for the rest).  Allreduce adds the mirror image: in round t
    unit i > 0 passes block t - (p - 1 - i) to unit i - 1, which overwrites.
    2 (p + m - 2) rounds for p >= 2.
    """
    sim = RankSim(bufs, arith)
    P, n = sim.P, sim.n
    if m < 1:
        raise ValueError("m must be at least 1")
    if P == 1:
        return sim.result()
    blocks = split(n, m)
    for t in range(P + m - 2):
        sim.round([(i, i + 1, *blocks[t - i], "add") for i in range(P - 1) if 0 <= t - i < m])
    for t in range(P + m - 2):
        sim.round([(i, i - 1, *blocks[t - (P - 1 - i)], "copy") for i in range(1, P)
                   if 0 <= t - (P - 1 - i) < m])
    return sim.result()


def ahc_layout(group_sizes):
    """AHC chunking: LCM of the group sizes, G groups, LCM x G chunks; group
    offsets (groups are contiguous rank ranges in the given order)."""
    sizes = [int(g) for g in group_sizes]
    if not sizes or min(sizes) < 1:
        raise ValueError("AHC needs at least one group, every group non-empty")
    M = 1
    for g in sizes:
        M = M * g // math.gcd(M, g)
    G = len(sizes)
    offs = [0]
    for g in sizes:
        offs.append(offs[-1] + g)
    return M, G, M * G, offs


def ahc_holder(group_sizes, offs, M, gamma, k):
    """Rank holding logical device k in group gamma after the intra-group
    reduce-scatter: the part containing the logical device's chunks is
    floor(k g / M), and the ring reduce-scatter leaves part p on member p - 1."""
    g = group_sizes[gamma]
    part = (k * g) // M
    return offs[gamma] + (part - 1) % g


def ahc(bufs, arith, group_sizes):
    """AHC hierarchical allreduce (intra / inter / intra all by ring).

    1. Groups are contiguous rank ranges.  The data is cut into LCM x G chunks;
       each group runs a ring reduce-scatter (the ring above, over its g parts
       of LCM x G / g consecutive chunks), all groups in parallel.
    2. Logical device k = 0..LCM-1 owns chunks [kG, (k+1)G).  The ranks that
       hold it in each group are the logical devices with identical IDs; they
       run a ring allreduce over its G chunks, in group order.
    3. Each group runs a ring all-gather over its parts.
    """
    sim = RankSim(bufs, arith)
    P, n = sim.P, sim.n
    sizes = [int(g) for g in group_sizes]
    M, G, nch, offs = ahc_layout(sizes)
    if offs[-1] != P:
        raise ValueError("AHC group sizes must add up to P")
    ch = split(n, nch)

    def span(c0, c1):
        return _chunk_span(ch, c0, c1)

    gmax = max(sizes)
    for t in range(gmax - 1):
        msgs = []
        for gamma, g in enumerate(sizes):
            if t >= g - 1:
                continue
            w = nch // g
            for m in range(g):
                p = (m - t) % g
                msgs.append((offs[gamma] + m, offs[gamma] + (m + 1) % g,
                             *span(p * w, (p + 1) * w), "add"))
        sim.round(msgs)
    holders = [[ahc_holder(sizes, offs, M, gamma, k) for gamma in range(G)]
               for k in range(M)]
    for phase, kind in (("rs", "add"), ("ag", "copy")):
        for t in range(G - 1):
            msgs = []
            for k in range(M):
                hs = holders[k]
                for i in range(G):
                    j = (i - t) % G if phase == "rs" else (i + 1 - t) % G
                    c = k * G + j
                    msgs.append((hs[i], hs[(i + 1) % G], *span(c, c + 1), kind))
            sim.round(msgs)
    for t in range(gmax - 1):
        msgs = []
        for gamma, g in enumerate(sizes):
            if t >= g - 1:
                continue
            w = nch // g
            for m in range(g):
                p = (m + 1 - t) % g
                msgs.append((offs[gamma] + m, offs[gamma] + (m + 1) % g,
                             *span(p * w, (p + 1) * w), "copy"))
        sim.round(msgs)
    info = {"lcm": M, "groups": G, "chunks": nch, "holders": holders}
    return sim.result(info)


def run(algo, bufs, arith, group="cyclic", r=0, k1=0, group_sizes=None, blocks=1, phase="allreduce"):
    """Run one schedule by name; phase picks a half of the splitting ones.

    avg runs the schedule as a sum and divides every finished sum by P once
    (a copy of a finished sum carries the divided value, so dividing where
    each sum completes or every rank's result at the end is the same); an
    all-gather combines nothing and divides nothing.
    """
    if phase != "allreduce" and algo not in ("ring", "rh", "generalized"):
        raise ValueError(f"{algo} does not split into a reduce-scatter and an all-gather")
    res = _run(algo, bufs, arith, group, r, k1, group_sizes, blocks, phase)
    if getattr(arith, "op", None) == "avg" and phase != "all_gather":
        P = len(bufs)
        if phase == "allreduce":
            res.bufs = [arith.average(b, P) for b in res.bufs]
        else:
            # the owners' chunks are the finished sums of a reduce-scatter
            for rank, lo, hi in res.info["owner"]:
                res.bufs[rank][lo:hi] = arith.average(res.bufs[rank][lo:hi], P)
    return res


def _run(algo, bufs, arith, group, r, k1, group_sizes, blocks, phase):
    if algo == "ring":
        return ring(bufs, arith, phase)
    if algo == "binomial":
        return binomial(bufs, arith)
    if algo == "rd":
        return rd(bufs, arith)
    if algo == "rh":
        return rh(bufs, arith, phase)
    if algo == "hybrid":
        return hybrid(bufs, arith, k1)
    if algo == "generalized":
        return generalized(bufs, arith, group, r, phase)
    if algo == "ahc":
        return ahc(bufs, arith, group_sizes)
    if algo == "pipeline":
        return pipeline(bufs, arith, blocks)
    raise ValueError(f"unknown algorithm {algo!r}")
