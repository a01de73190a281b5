// Schedule compiler.  Each generator below emits the rounds of one schedule as
// transfers between (rank, slot) storage over element ranges; run_symbolic()
// then executes the rounds on reduction-tree ids instead of values, which
// yields for every element of every rank the exact tree the schedule builds.
// The tile programs of both kernel forms are derived from these two results.

#include "schedule.hpp"

#include <algorithm>
#include <map>
#include <numeric>
#include <set>
#include <stdexcept>
#include <tuple>

namespace ar {

int32_t Dag::combine(int32_t l, int32_t r) {
    uint64_t key = (static_cast<uint64_t>(static_cast<uint32_t>(l)) << 32) | static_cast<uint32_t>(r);
    auto it = memo_.find(key);
    if (it != memo_.end()) return it->second;
    int32_t id = size();
    kids_.push_back(l);
    kids_.push_back(r);
    memo_.emplace(key, id);
    return id;
}

std::string Dag::text(int32_t x) const {
    if (leaf(x)) return std::to_string(x);
    return "(" + text(left(x)) + "+" + text(right(x)) + ")";
}

bool Dag::complete(int32_t x) const {
    // leaf multiset by an explicit stack (trees have at most P leaves)
    std::vector<int> count(P_, 0);
    std::vector<int32_t> stack{x};
    int total = 0;
    while (!stack.empty()) {
        int32_t y = stack.back();
        stack.pop_back();
        if (leaf(y)) {
            if (++count[y] > 1) return false;
            if (++total > P_) return false;
        } else {
            stack.push_back(left(y));
            stack.push_back(right(y));
        }
    }
    return total == P_;
}

int Schedule::seg_of(int64_t elem) const {
    auto it = std::upper_bound(bounds.begin(), bounds.end(), elem);
    return static_cast<int>(it - bounds.begin()) - 1;
}

std::vector<std::pair<int64_t, int64_t>> ceil_split(int64_t n, int64_t N) {
    // ceil chunk split: parts of ceil(n / N) elements, the last ones short or
    // empty ("All-Reduce, in depth", The ring algorithm, the split helper).
    std::vector<std::pair<int64_t, int64_t>> out;
    int64_t size = n > 0 ? (n + N - 1) / N : 0;
    for (int64_t k = 0; k < N; ++k)
        out.emplace_back(std::min(n, k * size), std::min(n, (k + 1) * size));
    return out;
}

int ceil_log2(int64_t P) {
    int L = 0;
    while ((int64_t(1) << L) < P) ++L;
    return L;
}

int esize_of(int dtype) { return dtype == AR_BFLOAT16 ? 2 : 4; }

namespace {

bool is_pow2(int P) { return P >= 1 && (P & (P - 1)) == 0; }
int mod(int64_t a, int64_t m) { return static_cast<int>(((a % m) + m) % m); }

struct Gen {
    Schedule& S;
    int P;        // ranks taking part (0..P-1)
    int64_t n;
    int P_total;  // ranks of the whole schedule (size of the sent counters)
    int phase;    // AR_PHASE_*: both halves, or the reduce-scatter / all-gather half
    bool rs() const { return phase != AR_PHASE_ALL_GATHER; }
    bool ag() const { return phase != AR_PHASE_REDUCE_SCATTER; }

    Round& new_round() {
        S.rounds.emplace_back();
        S.rounds.back().sent.assign(P_total, 0);
        return S.rounds.back();
    }
    // A plain message: one transfer whose bytes count as sent by src.
    void msg(Round& rd, int src, int dst, int64_t lo, int64_t hi, bool combine) {
        rd.sent[src] += hi - lo;
        if (hi > lo) rd.xfers.push_back({src, 0, dst, 0, 0, lo, hi, combine});
    }
};

// Ring reduce-scatter + all-gather ("All-Reduce, in depth", The ring
// algorithm): round t of the reduce-scatter has rank r pass chunk (r - t) mod P
// to r + 1, which adds it into its copy; round t of the all-gather has rank r
// pass chunk (r + 1 - t) mod P on, overwriting.
void gen_ring(Gen& g) {
    auto ch = ceil_split(g.n, g.P);
    for (int t = 0; g.rs() && t + 1 < g.P; ++t) {
        Round& rd = g.new_round();
        for (int r = 0; r < g.P; ++r) {
            auto c = ch[mod(r - t, g.P)];
            g.msg(rd, r, (r + 1) % g.P, c.first, c.second, true);
        }
    }
    for (int t = 0; g.ag() && t + 1 < g.P; ++t) {
        Round& rd = g.new_round();
        for (int r = 0; r < g.P; ++r) {
            auto c = ch[mod(r + 1 - t, g.P)];
            g.msg(rd, r, (r + 1) % g.P, c.first, c.second, false);
        }
    }
}

// Binomial tree ("還元演算子", binomial tree): in round k every active unit with
// bit k set hands its vector to the unit 2^k below and retires; an active
// unit i with i + 2^k < P combines x_i <- x_i (+) x_{i+2^k}.  The broadcast
// from unit 0 runs the tree backwards with copies.
void gen_binomial(Gen& g) {
    int L = ceil_log2(g.P);
    std::vector<bool> active(g.P, true);
    for (int k = 0; k < L; ++k) {
        Round& rd = g.new_round();
        for (int i = 0; i < g.P; ++i) {
            if (!active[i]) continue;
            if ((i >> k) & 1) {
                active[i] = false;
            } else if (i + (1 << k) < g.P) {
                g.msg(rd, i + (1 << k), i, 0, g.n, true);
            }
        }
    }
    for (int k = L - 1; k >= 0; --k) {
        Round& rd = g.new_round();
        for (int i = 0; i + (1 << k) < g.P; i += 1 << (k + 1)) g.msg(rd, i, i + (1 << k), 0, g.n, false);
    }
}

// Recursive doubling over [lo, hi) with distances 1, 2, ..., 2^(steps-1):
// every rank combines the partner's pre-round block into its own.
void rd_rounds(Gen& g, int steps, const std::vector<std::pair<int64_t, int64_t>>& block) {
    for (int k = 0; k < steps; ++k) {
        Round& rd = g.new_round();
        int d = 1 << k;
        for (int r = 0; r < g.P; ++r) g.msg(rd, r ^ d, r, block[r].first, block[r].second, true);
    }
}

// Classic hybrid: k1 halving rounds (distance P/2 first, each rank keeps the
// half of its chunk range whose bit matches its own and sends the other half
// to the partner), recursive doubling on the block each rank then owns, and
// the k1 mirrored doubling rounds (copies).
void gen_hybrid(Gen& g, int k1) {
    int L = ceil_log2(g.P);
    auto ch = ceil_split(g.n, g.P);
    std::vector<std::pair<int, int>> own(g.P, {0, g.P});
    auto span = [&](std::pair<int, int> cr) {
        return std::make_pair(ch[cr.first].first, ch[cr.second - 1].second);
    };
    for (int i = 0; i < k1; ++i) {
        Round& rd = g.new_round();
        int d = g.P >> (i + 1);
        std::vector<std::pair<int, int>> nxt(g.P);
        for (int r = 0; r < g.P; ++r) {
            int c0 = own[r].first, c1 = own[r].second, mid = (c0 + c1) / 2;
            std::pair<int, int> keep = (r & d) ? std::make_pair(mid, c1) : std::make_pair(c0, mid);
            std::pair<int, int> give = (r & d) ? std::make_pair(c0, mid) : std::make_pair(mid, c1);
            auto e = span(give);
            g.msg(rd, r, r ^ d, e.first, e.second, true);
            nxt[r] = keep;
        }
        own = nxt;
    }
    std::vector<std::pair<int64_t, int64_t>> block(g.P);
    for (int r = 0; r < g.P; ++r) block[r] = span(own[r]);
    rd_rounds(g, L - k1, block);
    for (int i = k1 - 1; i >= 0; --i) {
        Round& rd = g.new_round();
        int d = g.P >> (i + 1);
        for (int r = 0; r < g.P; ++r) {
            auto e = span(own[r]);
            g.msg(rd, r, r ^ d, e.first, e.second, false);
        }
        std::vector<std::pair<int, int>> nxt(g.P);
        for (int r = 0; r < g.P; ++r)
            nxt[r] = {std::min(own[r].first, own[r ^ d].first), std::max(own[r].second, own[r ^ d].second)};
        own = nxt;
    }
}

int pow2_floor(int P) {
    int Pp = 1;
    while (Pp * 2 <= P) Pp *= 2;
    return Pp;
}

// Any P for a power-of-two schedule ("A Generalization of the Allreduce
// Operation", introduction: reduce the process count to the largest power of
// two P' with a preparation and a finalization step).  Preparation: excess
// rank P' + i sends its vector to rank i, which combines it.  The inner
// schedule then runs on ranks 0..P'-1 (chunked over P').  Finalization: rank
// i sends the result back to rank P' + i.
template <class Inner>
void gen_fold(Gen& g, Inner inner) {
    const int Pp = pow2_floor(g.P);
    if (Pp == g.P) {
        inner(g);
        return;
    }
    const int e = g.P - Pp;
    if (g.rs()) {
        Round& rd = g.new_round();
        for (int i = 0; i < e; ++i) g.msg(rd, Pp + i, i, 0, g.n, true);
    }
    Gen h{g.S, Pp, g.n, g.P_total, g.phase};
    inner(h);
    if (g.ag()) {
        Round& rd = g.new_round();
        for (int i = 0; i < e; ++i) g.msg(rd, i, Pp + i, 0, g.n, false);
    }
}

// Generalized allreduce ("A Generalization of the Allreduce Operation",
// eqs. 17-44), positions model.  Position a's distributed vector keeps chunk
// c on rank t_a(c) (cyclic: a + c mod P; XOR: a ^ c).  Reduction step i with
// N = N_i, h = floor(N/2), lo = N - 2h: the vectors at positions lo+h..N-1 move
// by -h and combine into positions lo..lo+h-1; position 0 idles when N is odd.
// Removing r distribution steps runs T = N_{L-r} targets, target s shifting
// every position by s.  Identical (position, partial) pairs are one message
// and identical results one combine.  A rank keeps each distinct live
// partial of a chunk in its own slot (slot 0 = its buffer).
void gen_generalized(Gen& g, bool xr, int r) {
    const int P = g.P;
    auto ch = ceil_split(g.n, P);
    std::vector<int> Ns{P};
    while (Ns.back() > 1) Ns.push_back((Ns.back() + 1) / 2);
    const int L = static_cast<int>(Ns.size()) - 1;
    const int T = Ns[L - r];
    auto comp = [&](int s, int j) { return xr ? (s ^ j) : (s + j) % P; };
    auto rank_of = [&](int a, int c) { return xr ? (a ^ c) : (a + c) % P; };
    auto shift = [&](int a, int h) { return xr ? (a ^ h) : (a + h) % P; };

    // partial trees over vector indices (leaf v = vector v)
    Dag vt(P);
    std::vector<std::vector<int32_t>> cur(T, std::vector<int32_t>(P));
    for (int s = 0; s < T; ++s)
        for (int j = 0; j < P; ++j) cur[s][j] = comp(s, j);
    // slot -> partial per absolute position (-1 = free)
    std::vector<std::vector<int32_t>> slots(P);
    for (int a = 0; a < P; ++a) slots[a] = {a};
    auto slot_of = [&](int a, int32_t t) {
        for (size_t k = 0; k < slots[a].size(); ++k)
            if (slots[a][k] == t) return static_cast<int>(k);
        throw std::logic_error("generalized: partial not resident");
    };

    for (int i = 0; g.rs() && i < L; ++i) {
        const int N = Ns[i], h = N / 2, lo = N - 2 * h;
        std::set<std::pair<int, int32_t>> msgs;
        // (a_dst, t_new) -> (t_dst, a_src, t_src)
        std::map<std::pair<int, int32_t>, std::tuple<int32_t, int, int32_t>> combos;
        std::vector<std::vector<int32_t>> nxt(T);
        for (int s = 0; s < T; ++s) nxt[s].assign(cur[s].begin(), cur[s].begin() + Ns[i + 1]);
        for (int s = 0; s < T; ++s) {
            for (int j = lo; j < lo + h; ++j) {
                int a_dst = comp(s, j), a_src = comp(s, j + h);
                int32_t t_dst = cur[s][j], t_src = cur[s][j + h];
                int32_t t_new = vt.combine(t_dst, t_src);
                msgs.insert({a_src, t_src});
                combos[{a_dst, t_new}] = {t_dst, a_src, t_src};
                nxt[s][j] = t_new;
            }
        }
        // live partials after the step, per position
        std::vector<std::set<int32_t>> live(P);
        for (int s = 0; s < T; ++s)
            for (int j = 0; j < Ns[i + 1]; ++j) live[comp(s, j)].insert(nxt[s][j]);
        // slot assignment: carried partials keep their slot, new ones take the
        // lowest free slot
        std::vector<std::vector<int32_t>> new_slots(P);
        std::map<std::pair<int, int32_t>, int> out_slot;
        for (int a = 0; a < P; ++a) {
            std::vector<int32_t> ns(slots[a].size(), -1);
            for (size_t k = 0; k < slots[a].size(); ++k)
                if (slots[a][k] >= 0 && live[a].count(slots[a][k])) ns[k] = slots[a][k];
            for (auto& kv : combos) {
                if (kv.first.first != a) continue;
                size_t k = 0;
                while (k < ns.size() && ns[k] != -1) ++k;
                if (k == ns.size()) ns.push_back(-1);
                ns[k] = kv.first.second;
                out_slot[kv.first] = static_cast<int>(k);
            }
            new_slots[a] = ns;
        }
        Round& rd = g.new_round();
        for (auto& kv : combos) {
            int a_dst = kv.first.first;
            int32_t t_dst, t_src;
            int a_src;
            std::tie(t_dst, a_src, t_src) = kv.second;
            int ss = slot_of(a_src, t_src), sd = slot_of(a_dst, t_dst), so = out_slot[kv.first];
            for (int c = 0; c < P; ++c) {
                if (ch[c].second <= ch[c].first) continue;
                rd.xfers.push_back({rank_of(a_src, c), ss, rank_of(a_dst, c), sd, so, ch[c].first,
                                    ch[c].second, true});
            }
        }
        for (auto& m : msgs)
            for (int c = 0; c < P; ++c) rd.sent[rank_of(m.first, c)] += ch[c].second - ch[c].first;
        slots = new_slots;
        cur = nxt;
    }
    // every target's result sits in slot 0 of its position (its last combine
    // found the old slots dead); the distribution copies slot 0 to slot 0
    for (int a = 0; a < T; ++a)
        if (slot_of(a, cur[a][0]) != 0) throw std::logic_error("generalized: result not in slot 0");
    for (int i = L - r - 1; g.ag() && i >= 0; --i) {
        const int N = Ns[i], h = N / 2, lo = N - 2 * h;
        Round& rd = g.new_round();
        for (int a = lo; a < lo + h; ++a) {
            int b = shift(a, h);
            for (int c = 0; c < P; ++c) {
                if (ch[c].second <= ch[c].first) continue;
                rd.xfers.push_back({rank_of(a, c), 0, rank_of(b, c), 0, 0, ch[c].first, ch[c].second, false});
                rd.sent[rank_of(a, c)] += ch[c].second - ch[c].first;
            }
        }
    }
}

// AHC (HCCL, Description): contiguous groups, LCM x G chunks; ring
// reduce-scatter inside every group over its g parts (groups in parallel);
// logical device k owns chunks [kG, (k+1)G) and is held in each group by the
// member the reduce-scatter left its part on; those holders run a ring
// allreduce over the G chunks; ring all-gather inside every group.
void gen_ahc(Gen& g, const std::vector<int>& sizes) {
    int64_t M = 1;
    for (int s : sizes) M = M / std::gcd(M, static_cast<int64_t>(s)) * s;
    const int G = static_cast<int>(sizes.size());
    const int64_t nch = M * G;
    auto ch = ceil_split(g.n, nch);
    std::vector<int> offs{0};
    for (int s : sizes) offs.push_back(offs.back() + s);
    auto span = [&](int64_t c0, int64_t c1) { return std::make_pair(ch[c0].first, ch[c1 - 1].second); };
    int gmax = *std::max_element(sizes.begin(), sizes.end());
    auto intra = [&](bool combine) {
        for (int t = 0; t + 1 < gmax; ++t) {
            Round& rd = g.new_round();
            for (int gm = 0; gm < G; ++gm) {
                int gs = sizes[gm];
                if (t >= gs - 1) continue;
                int64_t w = nch / gs;
                for (int m = 0; m < gs; ++m) {
                    int p = combine ? mod(m - t, gs) : mod(m + 1 - t, gs);
                    auto e = span(p * w, (p + 1) * w);
                    g.msg(rd, offs[gm] + m, offs[gm] + (m + 1) % gs, e.first, e.second, combine);
                }
            }
        }
    };
    intra(true);
    std::vector<std::vector<int>> holders(M, std::vector<int>(G));
    for (int64_t k = 0; k < M; ++k)
        for (int gm = 0; gm < G; ++gm) {
            int gs = sizes[gm];
            int part = static_cast<int>((k * gs) / M);
            holders[k][gm] = offs[gm] + mod(part - 1, gs);
        }
    for (int phase = 0; phase < 2; ++phase) {
        for (int t = 0; t + 1 < G; ++t) {
            Round& rd = g.new_round();
            for (int64_t k = 0; k < M; ++k) {
                for (int i = 0; i < G; ++i) {
                    int j = phase == 0 ? mod(i - t, G) : mod(i + 1 - t, G);
                    auto e = span(k * G + j, k * G + j + 1);
                    g.msg(rd, holders[k][i], holders[k][(i + 1) % G], e.first, e.second, phase == 0);
                }
            }
        }
    }
    intra(false);
}

// Pipelined chain reduce ("還元演算子", pipelined algorithm): m blocks; round
// t has unit i pass block t - i to unit i + 1, which combines it, so the last
// unit has every block after p + m - 2 rounds; the broadcast mirrors it (unit
// i passes block t - (p - 1 - i) to unit i - 1, which overwrites).
void gen_pipeline(Gen& g, int m) {
    if (g.P < 2) return;
    auto blk = ceil_split(g.n, m);
    for (int t = 0; t < g.P + m - 2; ++t) {
        Round& rd = g.new_round();
        for (int i = 0; i + 1 < g.P; ++i)
            if (t - i >= 0 && t - i < m) g.msg(rd, i, i + 1, blk[t - i].first, blk[t - i].second, true);
    }
    for (int t = 0; t < g.P + m - 2; ++t) {
        Round& rd = g.new_round();
        for (int i = 1; i < g.P; ++i) {
            const int b = t - (g.P - 1 - i);
            if (b >= 0 && b < m) g.msg(rd, i, i - 1, blk[b].first, blk[b].second, false);
        }
    }
}

// Runs the rounds on tree ids: every transfer reads the pre-round state, a
// round may write each (rank, slot, segment) once, combines intern
// (receiver, incoming) in the DAG.
void run_symbolic(Schedule& S) {
    std::vector<int64_t> b{0, S.n};
    int max_slot = 0;
    for (auto& rd : S.rounds)
        for (auto& x : rd.xfers) {
            b.push_back(x.lo);
            b.push_back(x.hi);
            max_slot = std::max({max_slot, x.src_slot, x.dst_in, x.dst_out});
        }
    std::sort(b.begin(), b.end());
    b.erase(std::unique(b.begin(), b.end()), b.end());
    S.bounds = b;
    S.max_slots = max_slot + 1;
    const int nseg = S.nseg(), P = S.P, ns = S.max_slots;
    S.dag = Dag(P);
    std::vector<int32_t> state(static_cast<size_t>(P) * ns * nseg, -1);
    auto at = [&](int rank, int slot, int seg) -> int32_t& {
        return state[(static_cast<size_t>(rank) * ns + slot) * nseg + seg];
    };
    for (int r = 0; r < P; ++r)
        for (int s = 0; s < nseg; ++s) at(r, 0, s) = r;
    std::vector<int32_t> stamp(state.size(), -1);
    S.combines = 0;
    for (size_t ri = 0; ri < S.rounds.size(); ++ri) {
        std::vector<std::pair<size_t, int32_t>> writes;
        for (auto& x : S.rounds[ri].xfers) {
            int s0 = S.seg_of(x.lo), s1 = S.seg_of(x.hi - 1) + 1;
            if (x.combine && S.op == AR_AVG) x.completes.assign(s1 - s0, 0);
            for (int s = s0; s < s1; ++s) {
                int32_t v = at(x.src, x.src_slot, s);
                if (v < 0) throw std::logic_error("schedule reads an empty slot");
                if (x.combine) {
                    int32_t d = at(x.dst, x.dst_in, s);
                    if (d < 0) throw std::logic_error("schedule combines into an empty slot");
                    v = S.dag.combine(d, v);
                    if (S.op == AR_AVG) x.completes[s - s0] = S.dag.complete(v);
                }
                size_t idx = (static_cast<size_t>(x.dst) * ns + x.dst_out) * nseg + s;
                if (stamp[idx] == static_cast<int32_t>(ri)) throw std::logic_error("round writes a slot twice");
                stamp[idx] = static_cast<int32_t>(ri);
                writes.emplace_back(idx, v);
            }
            if (x.combine) S.combines += x.hi - x.lo;
        }
        for (auto& w : writes) state[w.first] = w.second;
    }
    S.final_node.assign(static_cast<size_t>(P) * nseg, -1);
    S.defined.assign(static_cast<size_t>(P) * nseg, 0);
    const int phase = S.params.phase;
    for (int s = 0; s < nseg; ++s) {
        const bool empty = S.bounds[s + 1] <= S.bounds[s];
        int owners = 0;
        for (int r = 0; r < P; ++r) {
            const int32_t v = at(r, 0, s);
            const size_t k = static_cast<size_t>(r) * nseg + s;
            S.final_node[k] = v;
            if (phase == AR_PHASE_ALLREDUCE) {
                if (!empty && !S.dag.complete(v)) throw std::logic_error("schedule leaves an incomplete reduction");
                S.defined[k] = 1;
            } else if (phase == AR_PHASE_REDUCE_SCATTER) {
                S.defined[k] = S.dag.complete(v);
                owners += S.defined[k];
            } else {
                // all-gather: every rank ends with the owner's own value
                if (!empty && (!S.dag.leaf(v) || v != at(0, 0, s)))
                    throw std::logic_error("all-gather leaves ranks disagreeing");
                S.defined[k] = v != r;
            }
        }
        if (phase == AR_PHASE_REDUCE_SCATTER && !empty && owners == 0)
            throw std::logic_error("reduce-scatter leaves a chunk without an owner");
    }
}

}  // namespace

ar_status compile_schedule(int P, int64_t n, int dtype, int op, int algo, const ar_params* p,
                           Schedule& S) {
    if (P < 1 || n < 0) return AR_ERR_INVALID_ARG;
    if (dtype < AR_INT32 || dtype > AR_BFLOAT16) return AR_ERR_INVALID_ARG;
    if (op < AR_SUM || op > AR_AVG) return AR_ERR_INVALID_ARG;
    if (op == AR_AVG && dtype == AR_INT32) return AR_ERR_UNSUPPORTED;
    if (algo < AR_RING || algo > AR_PIPELINE) return AR_ERR_INVALID_ARG;
    if (P > AR_MAX_RANKS) return AR_ERR_UNSUPPORTED;
    Params pr;
    if (p) {
        pr.form = p->form;
        pr.order = p->order;
        pr.group = p->group;
        pr.r = p->r;
        pr.k1 = p->k1;
        pr.blocks = p->blocks == 0 ? 1 : p->blocks;
        pr.phase = p->phase;
        pr.jit = p->jit;
        if (algo == AR_AHC) {
            if (p->n_groups < 1 || !p->group_sizes) return AR_ERR_INVALID_ARG;
            pr.group_sizes.assign(p->group_sizes, p->group_sizes + p->n_groups);
        }
    } else if (algo == AR_AHC) {
        return AR_ERR_INVALID_ARG;
    }
    if (pr.form != AR_FORM_FUSED && pr.form != AR_FORM_STEP) return AR_ERR_INVALID_ARG;
    if (pr.order != AR_ORDER_FAITHFUL && pr.order != AR_ORDER_FP32ACC) return AR_ERR_INVALID_ARG;
    if (pr.group != AR_GROUP_CYCLIC && pr.group != AR_GROUP_XOR) return AR_ERR_INVALID_ARG;
    if (pr.form == AR_FORM_STEP && pr.order == AR_ORDER_FP32ACC) return AR_ERR_UNSUPPORTED;
    if (pr.phase < AR_PHASE_ALLREDUCE || pr.phase > AR_PHASE_ALL_GATHER) return AR_ERR_INVALID_ARG;
    if (pr.jit < AR_JIT_OFF || pr.jit > AR_JIT_ON) return AR_ERR_INVALID_ARG;
    // the halves exist for the schedules that split into a reduce-scatter and
    // an all-gather: the ring, RH and the bandwidth-optimal generalized one
    if (pr.phase != AR_PHASE_ALLREDUCE) {
        const bool split = algo == AR_RING || algo == AR_RH || (algo == AR_GENERALIZED && pr.r == 0);
        if (!split) return AR_ERR_UNSUPPORTED;
        if (pr.phase == AR_PHASE_ALL_GATHER && pr.order == AR_ORDER_FP32ACC) return AR_ERR_UNSUPPORTED;
    }
    const int L = ceil_log2(P);
    const bool pow2 = is_pow2(P);
    switch (algo) {
        case AR_HYBRID:
            // any P: the halving steps run among the largest power of two
            if (pr.k1 < 0 || pr.k1 > ceil_log2(pow2_floor(P))) return AR_ERR_INVALID_ARG;
            break;
        case AR_PIPELINE:
            if (pr.blocks < 1 || pr.blocks > 4096) return AR_ERR_INVALID_ARG;
            break;
        case AR_GENERALIZED:
            if (pr.r < 0 || pr.r > L) return AR_ERR_INVALID_ARG;
            if (pr.group == AR_GROUP_XOR && !pow2) return AR_ERR_UNSUPPORTED;
            break;
        case AR_AHC: {
            int64_t sum = 0, M = 1;
            for (int s : pr.group_sizes) {
                if (s < 1) return AR_ERR_INVALID_ARG;
                sum += s;
                M = M / std::gcd(M, static_cast<int64_t>(s)) * s;
                if (M > 4096) return AR_ERR_UNSUPPORTED;
            }
            if (sum != P) return AR_ERR_INVALID_ARG;
            if (M * static_cast<int64_t>(pr.group_sizes.size()) > 4096) return AR_ERR_UNSUPPORTED;
            break;
        }
        default:
            break;
    }
    S = Schedule();
    S.P = P;
    S.n = n;
    S.dtype = dtype;
    S.op = op;
    S.algo = algo;
    S.params = pr;
    Gen g{S, P, n, P, pr.phase};
    try {
        switch (algo) {
            case AR_RING: gen_ring(g); break;
            case AR_BINOMIAL: gen_binomial(g); break;
            case AR_RH: gen_fold(g, [](Gen& h) { gen_generalized(h, true, 0); }); break;
            case AR_RD: gen_fold(g, [](Gen& h) { gen_hybrid(h, 0); }); break;
            case AR_HYBRID: gen_fold(g, [&](Gen& h) { gen_hybrid(h, pr.k1); }); break;
            case AR_GENERALIZED: gen_generalized(g, pr.group == AR_GROUP_XOR, pr.r); break;
            case AR_AHC: gen_ahc(g, pr.group_sizes); break;
            case AR_PIPELINE: gen_pipeline(g, pr.blocks); break;
        }
        run_symbolic(S);
    } catch (const std::bad_alloc&) {
        return AR_ERR_NOMEM;
    } catch (const std::logic_error&) {
        return AR_ERR_UNSUPPORTED;
    }
    return AR_OK;
}

}  // namespace ar
