// Lowering: compiled schedule -> tile programs -> work items.
//
// Fused form: every segment's program reads the P contributions once and
// evaluates the DAG of trees the P ranks end with.  For sum / prod (and every
// int32 op) a (+) b and b (+) a are bit-identical on the GPU (IEEE add / mul
// are commutative and NaN results are canonical), so the DAG is first
// canonicalised under commutation, which lets identical trees that differ only
// in operand order share one evaluation.  max / min keep the operand order
// (they differ on +-0 and NaN).
//
// Step form: every round's transfers (receiver on the left), grouped so that
// independent transfers run as separate chains and transfers that read each
// other's destinations are versioned into twin copies (step_sets).
#include "lower.hpp"

#include <algorithm>
#include <functional>
#include <map>
#include <stdexcept>

// Most outputs per item for which the rank-streaming kernel stores results
// with TMA bulk copies from shared memory (more: 128-bit stores).
#ifndef AR_TMA_STORE_MAX_OUT
#define AR_TMA_STORE_MAX_OUT 4
#endif

// Deepest tree stack (tiles below the top) streamed with 32 KB rank tiles.
#ifndef AR_TREE_WIDE_SLOTS
#define AR_TREE_WIDE_SLOTS 4
#endif

// Pipeline depth of the rank-streaming kernel for chains and for fp32
// accumulation over 4-byte elements (the others use as many stages as
// shared memory holds).
#ifndef AR_CHAIN_STAGES_4B
#define AR_CHAIN_STAGES_4B 3
#endif
#ifndef AR_ACC_STAGES_4B
#define AR_ACC_STAGES_4B 5
#endif
// ... and for bf16 chains (one bf16x2 instruction per element pair)
// Trees whose stack has more than AR_TMEM_TREE_MIN_SLOTS entries keep it in
// tensor memory (AR_TMEM_TREES), on 32 KB tiles with AR_TMEM_TREE_STAGES
// stages.
#ifndef AR_TMEM_TREES
#define AR_TMEM_TREES 1
#endif
#ifndef AR_TMEM_TREE_MIN_SLOTS
#define AR_TMEM_TREE_MIN_SLOTS 3
#endif
#ifndef AR_TMEM_TREE_STAGES
#define AR_TMEM_TREE_STAGES 4
#endif
#ifndef AR_MIN_TILE
#define AR_MIN_TILE 6144
#endif
#ifndef AR_JIT_STAGE_TABLE
#define AR_JIT_STAGE_TABLE 1
#endif
#ifndef AR_COPY_KERNEL
#define AR_COPY_KERNEL 1
#endif
#ifndef AR_FEW_KERNEL
#define AR_FEW_KERNEL 1
#endif
#ifndef AR_FEW_TREES
#define AR_FEW_TREES 1
#endif
#ifndef AR_FEW_LONG
#define AR_FEW_LONG 1
#endif
#ifndef AR_FEW_LONG_MIN_BYTES
#define AR_FEW_LONG_MIN_BYTES (1536ull << 20)
#endif

#ifndef AR_JIT_GEOMETRY
#define AR_JIT_GEOMETRY 1
#endif
#ifndef AR_JIT_WORD_STAGES
#define AR_JIT_WORD_STAGES 3
#endif
constexpr int kStagesWord = 8;
#ifndef AR_CHAIN_STAGES_BF16
#define AR_CHAIN_STAGES_BF16 4
#endif
// bf16 fp32 accumulation: rank tile (bytes: 24 KB or 32 KB), pipeline depth
// and TMA-store epilogue
#ifndef AR_BF16_ACC_TILE
#define AR_BF16_ACC_TILE 24576
#endif
#ifndef AR_ACC_STAGES_BF16
#define AR_ACC_STAGES_BF16 7
#endif
static_assert(AR_BF16_ACC_TILE == 24576 || AR_BF16_ACC_TILE == 32768, "a rank tile some instantiation runs");
#ifndef AR_BF16_ACC_TMA
#define AR_BF16_ACC_TMA 1
#endif

namespace ar {
namespace {

struct Prog {
    uint8_t kind = PK_DAG;
    uint8_t flags = 0;
    uint16_t n_tmp = 0;
    std::vector<uint16_t> in, out;
    std::vector<uint32_t> ins;
    int stores() const {
        if (kind != PK_DAG) return static_cast<int>(out.size());
        int s = 0;
        for (uint32_t w : ins) s += (w >> 30) != INS_OP;
        return s;  // (TREE programs store to their outputs like CHAIN / ACC)
    }
};

class Builder {
public:
    explicit Builder(Lowered& lw) : lw_(lw) {}
    uint32_t add(const Prog& p) {
        if (p.in.size() > MAX_IN || p.n_tmp > MAX_TMP) throw std::length_error("program too large");
        std::vector<uint32_t> key{p.kind, p.flags, p.n_tmp, static_cast<uint32_t>(p.in.size()),
                                  static_cast<uint32_t>(p.out.size())};
        key.insert(key.end(), p.in.begin(), p.in.end());
        key.insert(key.end(), p.out.begin(), p.out.end());
        key.insert(key.end(), p.ins.begin(), p.ins.end());
        auto it = index_.find(key);
        if (it != index_.end()) return it->second;
        DevProg d{};
        d.kind = p.kind;
        d.flags = p.flags;
        d.n_in = static_cast<uint16_t>(p.in.size());
        d.n_tmp = p.n_tmp;
        d.n_out = static_cast<uint16_t>(p.out.size());
        d.n_ins = static_cast<uint32_t>(p.ins.size());
        d.in_off = static_cast<uint32_t>(lw_.refs.size());
        lw_.refs.insert(lw_.refs.end(), p.in.begin(), p.in.end());
        d.out_off = static_cast<uint32_t>(lw_.refs.size());
        lw_.refs.insert(lw_.refs.end(), p.out.begin(), p.out.end());
        d.ins_off = static_cast<uint32_t>(lw_.ins.size());
        lw_.ins.insert(lw_.ins.end(), p.ins.begin(), p.ins.end());
        uint32_t id = static_cast<uint32_t>(lw_.progs.size());
        lw_.progs.push_back(d);
        stores_.push_back(p.stores());
        index_.emplace(std::move(key), id);
        return id;
    }
    int stores(uint32_t id) const { return stores_[id]; }

private:
    Lowered& lw_;
    std::map<std::vector<uint32_t>, uint32_t> index_;
    std::vector<int> stores_;
};

// Canonical DAG: same trees, children of commutative combines ordered.
struct Canon {
    Dag c;
    std::vector<int32_t> memo;
    const Dag& src;
    bool commute;
    Canon(const Dag& s, bool cm) : c(s.P()), memo(s.size(), -1), src(s), commute(cm) {}
    int32_t get(int32_t x) {
        if (src.leaf(x)) return x;
        if (memo[x] >= 0) return memo[x];
        int32_t a = get(src.left(x)), b = get(src.right(x));
        if (commute && a > b) std::swap(a, b);
        return memo[x] = c.combine(a, b);
    }
};

bool right_chain(const Dag& d, int32_t x, std::vector<int32_t>& leaves) {
    leaves.clear();
    while (!d.leaf(x)) {
        if (!d.leaf(d.left(x))) return false;
        leaves.push_back(d.left(x));
        x = d.right(x);
    }
    leaves.push_back(x);
    std::reverse(leaves.begin(), leaves.end());
    return true;
}

bool left_chain(const Dag& d, int32_t x, std::vector<int32_t>& leaves) {
    leaves.clear();
    while (!d.leaf(x)) {
        if (!d.leaf(d.right(x))) return false;
        leaves.push_back(d.right(x));
        x = d.left(x);
    }
    leaves.push_back(x);
    std::reverse(leaves.begin(), leaves.end());
    return true;
}

// Straight-line code for the trees outs[k].second that ranks outs[k].first
// must end with; avg: combined results are divided by P as they are stored.
Prog dag_program(const Dag& d, const std::vector<std::pair<int, int32_t>>& outs, bool avg) {
    const int P = d.P();
    Prog p;
    p.kind = PK_DAG;
    // post-order of the internal nodes reachable from the outputs
    std::vector<int32_t> topo;
    std::map<int32_t, int> uses;  // operand uses by internal nodes
    std::map<int32_t, std::vector<int>> stores_of;
    std::vector<char> seen(d.size(), 0);
    std::vector<char> leaf_used(P, 0);
    for (const auto& ro : outs) {
        stores_of[ro.second].push_back(ro.first);
        std::vector<std::pair<int32_t, int>> st{{ro.second, 0}};
        while (!st.empty()) {
            auto& top = st.back();
            int32_t x = top.first;
            if (d.leaf(x)) {
                leaf_used[x] = 1;
                st.pop_back();
                continue;
            }
            if (seen[x] == 2) {
                st.pop_back();
                continue;
            }
            if (top.second == 0) {
                top.second = 1;
                seen[x] = 1;
                st.push_back({d.left(x), 0});
            } else if (top.second == 1) {
                top.second = 2;
                st.push_back({d.right(x), 0});
            } else {
                seen[x] = 2;
                topo.push_back(x);
                st.pop_back();
            }
        }
    }
    for (int32_t x : topo) {
        uses[d.left(x)]++;
        uses[d.right(x)]++;
    }
    std::map<int32_t, uint32_t> loc;
    for (int r = 0; r < P; ++r)
        if (leaf_used[r]) {
            loc[r] = static_cast<uint32_t>(p.in.size());
            p.in.push_back(static_cast<uint16_t>(buf_id(0, r)));
        }
    for (int32_t leaf = 0; leaf < P; ++leaf)
        if (stores_of.count(leaf))
            for (int r : stores_of[leaf]) p.ins.push_back(ins_store(loc[leaf], buf_id(0, r)));
    std::vector<char> tmp_busy;
    auto alloc = [&]() -> uint32_t {
        size_t k = 0;
        while (k < tmp_busy.size() && tmp_busy[k]) ++k;
        if (k == tmp_busy.size()) tmp_busy.push_back(0);
        tmp_busy[k] = 1;
        p.n_tmp = std::max<uint16_t>(p.n_tmp, static_cast<uint16_t>(tmp_busy.size()));
        return REF_TMP | static_cast<uint32_t>(k);
    };
    std::map<int32_t, int> left_uses = uses;
    for (size_t k = 0; k < topo.size(); ++k) {
        int32_t x = topo[k];
        int32_t l = d.left(x), r = d.right(x);
        uint32_t a = loc.at(l), b = loc.at(r);
        for (int32_t o : {l, r}) {
            if (d.leaf(o)) continue;
            if (--left_uses[o] == 0) {
                uint32_t ref = loc[o];
                if (ref != REF_ACC && (ref & REF_TMP)) tmp_busy[ref & 0x1FF] = 0;
            }
        }
        bool next_uses = k + 1 < topo.size() && (d.left(topo[k + 1]) == x || d.right(topo[k + 1]) == x);
        uint32_t dest;
        if (uses[x] == 0 || (uses[x] == 1 && next_uses))
            dest = REF_ACC;
        else
            dest = alloc();
        p.ins.push_back(ins_op(a, b, dest));
        loc[x] = dest;
        if (stores_of.count(x))
            for (int rr : stores_of[x]) p.ins.push_back(ins_store(dest, buf_id(0, rr), avg));
    }
    return p;
}

// Post-order of a single tree: leaves left to right, and after each leaf the
// number of combines that follow it; false if the stack gets deeper than
// kTreeDepth.
bool tree_program(const Dag& d, int32_t root, bool commute, std::vector<int32_t>& leaves,
                  std::vector<uint32_t>& combines, int& depth) {
    leaves.clear();
    combines.clear();
    // Stack entries a subtree needs.  With a commutative op the deeper child
    // is evaluated first (Sethi-Ullman order: a chain needs 2 entries, not
    // one per leaf); the combine then takes the operands swapped, which
    // gives the same bits.
    std::map<int32_t, int> memo;
    std::function<int(int32_t)> need = [&](int32_t x) -> int {
        if (d.leaf(x)) return 1;
        auto it = memo.find(x);
        if (it != memo.end()) return it->second;
        const int l = need(d.left(x)), r = need(d.right(x));
        const int v = commute ? std::max(std::max(l, r), std::min(l, r) + 1) : std::max(l, r + 1);
        return memo[x] = v;
    };
    depth = need(root);
    if (depth > kTreeDepth) return false;
    struct Frame {
        int32_t x;
        int state;
        bool swap;
    };
    std::vector<Frame> st{{root, 0, false}};
    while (!st.empty()) {
        Frame& top = st.back();
        const int32_t x = top.x;
        if (d.leaf(x)) {
            leaves.push_back(x);
            combines.push_back(0);
            st.pop_back();
        } else if (top.state == 0) {
            top.state = 1;
            top.swap = commute && need(d.right(x)) > need(d.left(x));
            const int32_t first = top.swap ? d.right(x) : d.left(x);
            st.push_back({first, 0, false});
        } else if (top.state == 1) {
            top.state = 2;
            const int32_t second = top.swap ? d.left(x) : d.right(x);
            st.push_back({second, 0, false});
        } else {
            ++combines.back();
            st.pop_back();
        }
    }
    return leaves.size() <= static_cast<size_t>(kTreeMaxLeaves);
}

// The ranks a fused pass writes in a segment (every rank for an allreduce).
std::vector<int> defined_ranks(const Schedule& S, int seg) {
    std::vector<int> out;
    for (int r = 0; r < S.P; ++r)
        if (S.defined_at(r, seg)) out.push_back(r);
    return out;
}

void set_outputs(Prog& p, const std::vector<int>& ranks, int P) {
    for (int r : ranks) p.out.push_back(static_cast<uint16_t>(buf_id(0, r)));
    if (static_cast<int>(ranks.size()) == P) p.flags = PF_OUT_ALL;  // ranks are 0..P-1 in order
}

Prog fused_program(Canon& cn, const Schedule& S, int seg, const std::vector<int>& ranks) {
    std::vector<std::pair<int, int32_t>> outs;
    for (int r : ranks) outs.push_back({r, cn.get(S.final_at(r, seg))});
    const int32_t x = outs[0].second;
    bool same = std::all_of(outs.begin(), outs.end(), [&](const std::pair<int, int32_t>& o) { return o.second == x; });
    // AR_AVG divides combined results (an all-gather's copies are not)
    const bool avg = S.op == AR_AVG;
    std::vector<int32_t> leaves;
    if (same && (right_chain(cn.c, x, leaves) || left_chain(cn.c, x, leaves))) {
        Prog p;
        p.kind = right_chain(cn.c, x, leaves) ? PK_CHAIN_R : PK_CHAIN_L;
        if (p.kind == PK_CHAIN_L) left_chain(cn.c, x, leaves);
        for (int32_t l : leaves) p.in.push_back(static_cast<uint16_t>(buf_id(0, l)));
        set_outputs(p, ranks, S.P);
        if (avg && !cn.c.leaf(x)) p.flags |= PF_AVG;
        return p;
    }
    std::vector<uint32_t> combines;
    int depth = 0;
    if (same && tree_program(cn.c, x, cn.commute, leaves, combines, depth)) {
        Prog p;
        p.kind = PK_TREE;
        for (int32_t l : leaves) p.in.push_back(static_cast<uint16_t>(buf_id(0, l)));
        // combine counts (< kTreeDepth), 4 bits per leaf, 8 per word
        p.ins.assign(kTreeCountWords, 0);
        for (size_t i = 0; i < combines.size(); ++i) p.ins[i / 8] |= combines[i] << (4 * (i % 8));
        p.n_tmp = static_cast<uint16_t>(depth - 1);  // stack entries below the top
        set_outputs(p, ranks, S.P);
        if (avg && !cn.c.leaf(x)) p.flags |= PF_AVG;
        return p;
    }
    return dag_program(cn.c, outs, avg);
}

Prog acc_program(int P, const std::vector<int>& ranks, bool avg) {
    Prog p;
    p.kind = PK_ACC;
    for (int r = 0; r < P; ++r) p.in.push_back(static_cast<uint16_t>(buf_id(0, r)));
    set_outputs(p, ranks, P);
    if (avg) p.flags |= PF_AVG;
    return p;
}

using XferAvg = std::pair<const Transfer*, bool>;

// Whether a combine's operands may be swapped without changing a bit.
bool commute_ok(const Schedule& S) {
    return S.dtype == AR_INT32 || S.op == AR_SUM || S.op == AR_PROD || S.op == AR_AVG;
}

// The transfers of one round over one segment, split into groups that can
// run as separate work items: a transfer that writes a buffer joins every
// transfer that reads it (all of a group's reads must happen before its
// writes, which one work item guarantees); transfers sharing only sources
// stay apart.
std::vector<std::vector<XferAvg>> round_components(const std::vector<XferAvg>& xs) {
    const int n = static_cast<int>(xs.size());
    std::vector<int> parent(n);
    for (int i = 0; i < n; ++i) parent[i] = i;
    std::function<int(int)> find = [&](int i) { return parent[i] == i ? i : parent[i] = find(parent[i]); };
    std::map<uint32_t, int> writer;
    for (int i = 0; i < n; ++i) writer[buf_id(xs[i].first->dst_out, xs[i].first->dst)] = i;
    auto join_reader = [&](int i, uint32_t buf) {
        auto it = writer.find(buf);
        if (it != writer.end()) parent[find(i)] = find(it->second);
    };
    for (int i = 0; i < n; ++i) {
        const Transfer& x = *xs[i].first;
        join_reader(i, buf_id(x.src_slot, x.src));
        if (x.combine) join_reader(i, buf_id(x.dst_in, x.dst));
    }
    std::map<int, std::vector<XferAvg>> groups;
    for (int i = 0; i < n; ++i) groups[find(i)].push_back(xs[i]);
    std::vector<std::vector<XferAvg>> out;
    for (auto& kv : groups) out.push_back(std::move(kv.second));
    return out;
}

// One round over one segment: each transfer with whether its combine
// completes an AR_AVG sum (that result is divided by P as it is stored).
// commute: combines that swap the same two operands (the exchange of
// recursive doubling) give one value, computed once for every output.
Prog round_program(std::vector<XferAvg> xa, bool commute) {
    std::sort(xa.begin(), xa.end(), [](const std::pair<const Transfer*, bool>& a,
                                       const std::pair<const Transfer*, bool>& b) {
        return std::make_pair(a.first->dst, a.first->dst_out) < std::make_pair(b.first->dst, b.first->dst_out);
    });
    std::vector<const Transfer*> xs;
    for (const auto& t : xa) xs.push_back(t.first);
    Prog p;
    if (commute && xs.size() > 1) {
        // every transfer combines the same two buffers, in either order
        const Transfer& x0 = *xs[0];
        const uint32_t a = buf_id(x0.src_slot, x0.src), c = buf_id(x0.dst_in, x0.dst);
        bool same = a != c;
        for (size_t k = 0; k < xa.size() && same; ++k) {
            const Transfer& x = *xs[k];
            const uint32_t s0 = buf_id(x.src_slot, x.src), d0 = buf_id(x.dst_in, x.dst);
            same = x.combine && xa[k].second == xa[0].second &&
                   ((s0 == a && d0 == c) || (s0 == c && d0 == a));
        }
        if (same && x0.combine) {
            p.kind = PK_CHAIN_R;
            p.in.push_back(static_cast<uint16_t>(a));
            p.in.push_back(static_cast<uint16_t>(c));
            for (const Transfer* x : xs) p.out.push_back(static_cast<uint16_t>(buf_id(x->dst_out, x->dst)));
            if (xa[0].second) p.flags |= PF_AVG;
            return p;
        }
    }
    if (xs.size() == 1) {  // one transfer: acc = src, then dst_in (+) acc
        const Transfer& x = *xs[0];
        p.kind = PK_CHAIN_R;
        p.in.push_back(static_cast<uint16_t>(buf_id(x.src_slot, x.src)));
        if (x.combine) p.in.push_back(static_cast<uint16_t>(buf_id(x.dst_in, x.dst)));
        p.out.push_back(static_cast<uint16_t>(buf_id(x.dst_out, x.dst)));
        if (xa[0].second) p.flags |= PF_AVG;
        return p;
    }
    p.kind = PK_DAG;
    std::map<uint16_t, uint32_t> idx;
    auto input = [&](int slot, int rank) {
        uint16_t b = static_cast<uint16_t>(buf_id(slot, rank));
        auto it = idx.find(b);
        if (it != idx.end()) return it->second;
        uint32_t k = static_cast<uint32_t>(p.in.size());
        p.in.push_back(b);
        idx[b] = k;
        return k;
    };
    for (const Transfer* x : xs) {
        if (x->combine) input(x->dst_in, x->dst);
        input(x->src_slot, x->src);
    }
    for (size_t k = 0; k < xs.size(); ++k) {
        const Transfer* x = xs[k];
        uint32_t out = buf_id(x->dst_out, x->dst);
        if (x->combine) {
            p.ins.push_back(ins_op(idx[static_cast<uint16_t>(buf_id(x->dst_in, x->dst))],
                                   idx[static_cast<uint16_t>(buf_id(x->src_slot, x->src))], REF_ACC));
            p.ins.push_back(ins_store(REF_ACC, out, xa[k].second));
        } else {
            p.ins.push_back(ins_store(idx[static_cast<uint16_t>(buf_id(x->src_slot, x->src))], out));
        }
    }
    return p;
}

struct Range {
    uint32_t prog;
    int64_t lo, hi;
};

// Elements per work item of a set: a whole tile, unless the set is one range
// (one program over every element: the fp32-accumulate pass) whose whole
// tiles leave fewer items than half the GPU's 152 SMs — then about one item
// per SM, at least 1 KB per rank tile (a multiple of V elements, so items
// stay 16-byte aligned).  Measured: P = 64 x 256 KiB fp32 accumulation went
// from 95 us (8 items) to 24 us; splitting the ring's per-chunk ranges the
// same way made it slower (smaller rank tiles of many more items).
constexpr int64_t kFewItems = 152 / 2;
constexpr int64_t kSpreadItems = 152;

int64_t item_elems(const std::vector<Range>& rs, int64_t tile_elems, int64_t V) {
    int64_t body = 0, items = 0;
    for (const Range& r : rs) {
        const int64_t a = (r.lo + V - 1) / V * V, e = r.hi / V * V;
        if (a < e) {
            body += e - a;
            items += (e - a + tile_elems - 1) / tile_elems;
        }
    }
    if (body <= 0 || items >= kFewItems || rs.size() != 1) return tile_elems;
    const int64_t want = (body + kSpreadItems - 1) / kSpreadItems;
    return std::min(tile_elems, std::max(1024 / (16 / V), (want + V - 1) / V * V));
}

// Most inputs of a program of a set.
int set_max_in(const Lowered& lw, const std::vector<Range>& rs) {
    int m = 1;
    for (const Range& r : rs) m = std::max<int>(m, lw.progs[r.prog].n_in);
    return m;
}

// Mean elements per range (segment) of a set.
int64_t mean_range(const std::vector<Range>& rs) {
    int64_t n = 0;
    for (const Range& r : rs) n += r.hi - r.lo;
    return rs.empty() ? 0 : n / static_cast<int64_t>(rs.size());
}

void push_range(std::vector<Range>& v, uint32_t prog, int64_t lo, int64_t hi) {
    if (hi <= lo) return;
    if (!v.empty() && v.back().prog == prog && v.back().hi == lo)
        v.back().hi = hi;
    else
        v.push_back({prog, lo, hi});
}

// Step form.  Each round, per segment, is split into groups of transfers
// that read each other's destinations (round_components).  A group of one
// transfer, or recursive doubling's commutative exchange, runs in place.
// Any other group (the cyclic rounds of the generalized schedule with removed
// steps) is versioned instead of co-located: each of its transfers reads the
// current copy of its sources and writes its destination to another copy of
// that buffer, so every transfer is an independent chain that streams.  A
// rank's result (slot 0) has three physical copies: its own buffer and two
// twins in the plan's scratch (slots S and 2S, S = max_slots); redirected
// writes alternate between the twins, and its last write goes back to the
// rank's own buffer whenever the current copy is a twin (nobody reads the
// stale home copy then).  A second partial (slot k >= 1) toggles between its
// slot and one twin (k + S).  Results that still end in a twin are copied
// home by one final round.
void step_sets(const Schedule& S, Builder& b, std::vector<std::vector<Range>>& sets, Lowered& lw) {
    const int P = S.P, ns = S.max_slots, nseg = S.nseg();
    auto key = [&](int rank, int slot, int seg) { return (static_cast<size_t>(rank) * ns + slot) * nseg + seg; };
    std::vector<int> loc(static_cast<size_t>(P) * ns * nseg);
    for (int r = 0; r < P; ++r)
        for (int sl = 0; sl < ns; ++sl)
            for (int sg = 0; sg < nseg; ++sg) loc[key(r, sl, sg)] = sl;
    // the round of the last write of every rank's own buffer, per segment
    std::vector<int> last(static_cast<size_t>(P) * nseg, -1);
    for (size_t ri = 0; ri < S.rounds.size(); ++ri)
        for (const Transfer& x : S.rounds[ri].xfers)
            if (x.dst_out == 0)
                for (int sg = S.seg_of(x.lo), s1 = S.seg_of(x.hi - 1) + 1; sg < s1; ++sg)
                    last[static_cast<size_t>(x.dst) * nseg + sg] = static_cast<int>(ri);
    int phys_max = ns - 1;
    const bool commute = commute_ok(S);
    for (size_t ri = 0; ri < S.rounds.size(); ++ri) {
        const Round& rd = S.rounds[ri];
        std::map<int, std::vector<XferAvg>> by_seg;
        for (const Transfer& x : rd.xfers) {
            int s0 = S.seg_of(x.lo), s1 = S.seg_of(x.hi - 1) + 1;
            for (int sg = s0; sg < s1; ++sg)
                by_seg[sg].push_back({&x, !x.completes.empty() && x.completes[sg - s0] != 0});
        }
        std::vector<Range> rs;
        std::vector<std::pair<size_t, int>> moves;  // copies written this round: (key, physical slot)
        for (auto& kv : by_seg) {
            const int sg = kv.first;
            for (auto& comp : round_components(kv.second)) {
                const bool versioned = comp.size() > 1 && round_program(comp, commute).kind == PK_DAG;
                std::vector<Transfer> phys;
                phys.reserve(comp.size());
                for (const XferAvg& xa : comp) {
                    const Transfer& x = *xa.first;
                    Transfer y = x;
                    y.src_slot = loc[key(x.src, x.src_slot, sg)];
                    y.dst_in = loc[key(x.dst, x.dst_in, sg)];
                    const int cur = loc[key(x.dst, x.dst_out, sg)];
                    int out = cur;
                    if (x.dst_out == 0 && last[static_cast<size_t>(x.dst) * nseg + sg] == static_cast<int>(ri) &&
                        cur != 0)
                        out = 0;
                    else if (versioned && x.dst_out == 0)
                        out = cur == ns ? 2 * ns : ns;  // alternate between the two twins, away from home
                    else if (versioned)
                        out = cur == x.dst_out ? x.dst_out + ns : x.dst_out;  // a partial: its slot or its twin
                    y.dst_out = out;
                    phys_max = std::max(phys_max, out);
                    moves.push_back({key(x.dst, x.dst_out, sg), out});
                    phys.push_back(y);
                }
                if (versioned) {
                    for (size_t k = 0; k < phys.size(); ++k)
                        push_range(rs, b.add(round_program({{&phys[k], comp[k].second}}, commute)), S.bounds[sg],
                                   S.bounds[sg + 1]);
                } else {
                    std::vector<XferAvg> pc;
                    for (size_t k = 0; k < phys.size(); ++k) pc.push_back({&phys[k], comp[k].second});
                    push_range(rs, b.add(round_program(pc, commute)), S.bounds[sg], S.bounds[sg + 1]);
                }
            }
        }
        for (const auto& m : moves) loc[m.first] = m.second;
        sets.push_back(rs);
    }
    // results left in a twin: one more round of copies home
    std::vector<Transfer> copies;
    for (int r = 0; r < P; ++r)
        for (int sg = 0; sg < nseg; ++sg)
            if (loc[key(r, 0, sg)] != 0 && S.bounds[sg + 1] > S.bounds[sg]) {
                Transfer c{};
                c.src = r;
                c.src_slot = loc[key(r, 0, sg)];
                c.dst = r;
                c.dst_in = 0;
                c.dst_out = 0;
                c.lo = S.bounds[sg];
                c.hi = S.bounds[sg + 1];
                c.combine = false;
                copies.push_back(c);
            }
    std::vector<Range> home;
    for (const Transfer& c : copies) {
        const int sg = S.seg_of(c.lo);
        push_range(home, b.add(round_program({{&c, false}}, commute)), S.bounds[sg], S.bounds[sg + 1]);
    }
    if (!home.empty()) sets.push_back(home);
    lw.phys_slots = phys_max + 1;
}

}  // namespace

int staged_smem_bytes(const Lowered& lw) {
    // the mbarrier area, then the stage tiles and the temporaries
    return kBarrierBytes + lw.tile_bytes * (lw.stages * lw.max_in + lw.max_tmp);
}

int stream_smem_bytes(const Lowered& lw) {
    return kBarrierBytes + lw.stream_tile * (lw.stream_stages + (lw.stream_tmem ? 0 : lw.stream_slots));
}

void lower(const Schedule& S, Lowered& lw, const LowerOptions& opt) {
    lw = Lowered();
    const int es = esize_of(S.dtype);
    const int V = 16 / es;  // elements per 16-byte vector
    Builder b(lw);
    std::vector<std::vector<Range>> sets;
    if (S.P > 1 && S.n > 0) {
        if (S.params.form == AR_FORM_FUSED) {
            std::vector<Range> rs;
            const bool commute = S.dtype == AR_INT32 || S.op == AR_SUM || S.op == AR_PROD || S.op == AR_AVG;
            Canon cn(S.dag, commute);
            // With two ranks the fp32 accumulation is the schedule's single
            // combine (fp32 op, one rounding) for sum, prod and every int32
            // op, bit for bit: run the faithful program, which streams the
            // wider tiles.
            const bool acc = S.params.order == AR_ORDER_FP32ACC &&
                             !(S.P == 2 && (S.dtype == AR_INT32 || S.op == AR_SUM || S.op == AR_PROD));
            std::vector<std::pair<int, Prog>> progs;
            bool any_dag = false;
            for (int s = 0; s < S.nseg(); ++s) {
                if (S.bounds[s + 1] <= S.bounds[s]) continue;
                const std::vector<int> ranks = defined_ranks(S, s);
                if (ranks.empty()) continue;  // (an all-gather owner-only segment)
                progs.push_back({s, acc ? acc_program(S.P, ranks, S.op == AR_AVG) : fused_program(cn, S, s, ranks)});
                any_dag |= progs.back().second.kind == PK_DAG;
            }
            for (auto& sp : progs) {
                // a pass with DAG programs does not stream: its single trees
                // become DAG programs too (the staged and word kernels run
                // chains and DAGs, not tree stacks)
                if (any_dag && sp.second.kind == PK_TREE) {
                    std::vector<std::pair<int, int32_t>> outs;
                    for (int r : defined_ranks(S, sp.first)) outs.push_back({r, cn.get(S.final_at(r, sp.first))});
                    sp.second = dag_program(cn.c, outs, S.op == AR_AVG);
                }
                push_range(rs, b.add(sp.second), S.bounds[sp.first], S.bounds[sp.first + 1]);
            }
            sets.push_back(rs);
        } else {
            step_sets(S, b, sets, lw);
        }
    }
    // A set whose programs are all chains, single trees or fp32
    // accumulations streams one rank tile at a time (rank-streaming kernel);
    // sets with a DAG program stage all of an item's input tiles at once
    // (staged kernel).
    std::vector<bool> stream(sets.size(), true);
    for (size_t k = 0; k < sets.size(); ++k)
        for (auto& r : sets[k])
            if (lw.progs[r.prog].kind == PK_DAG) stream[k] = false;
    // Small sets (<= 256 KB of traffic) run as one element-wise launch: every
    // item's inputs load at once, where streaming P rank tiles one after the
    // other would pay P memory latencies.  Sets of chains whose segments are
    // under 4 KB per rank (tiny rank tiles) stage all of an item's tiles for
    // the same reason.
    std::vector<bool> small(sets.size(), false);
    for (size_t k = 0; k < sets.size(); ++k) {
        uint64_t bytes = 0;
        bool trees = false;
        for (auto& r : sets[k]) {
            const DevProg& d = lw.progs[r.prog];
            bytes += static_cast<uint64_t>(d.n_in + b.stores(r.prog)) * (r.hi - r.lo) * es;
            trees |= d.kind == PK_TREE;
        }
        small[k] = !sets[k].empty() && bytes <= (256u << 10);
        if (stream[k] && !small[k] && !trees && mean_range(sets[k]) * es < 4096) stream[k] = false;
    }
    // Sets with DAG programs of many inputs run on the word kernel when it is
    // available: its threads keep one 32-bit word of every input in registers,
    // where the staged kernel's shared memory holds ever smaller tiles as the
    // input count grows.
    std::vector<bool> words(sets.size(), false);
    for (size_t k = 0; k < sets.size(); ++k) {
        if (!opt.word_dag || stream[k] || small[k]) continue;
        int dag_in = 0;
        uint64_t bytes = 0;
        for (auto& r : sets[k]) {
            const DevProg& d = lw.progs[r.prog];
            if (d.kind == PK_DAG) dag_in = std::max<int>(dag_in, d.n_in);
            bytes += static_cast<uint64_t>(d.n_in + b.stores(r.prog)) * (r.hi - r.lo) * es;
        }
        words[k] = dag_in >= opt.word_min_in && dag_in > 0 && bytes >= opt.word_min_bytes;
    }
    // Fused chain passes of up to AR_CHAIN_WORD_MAX_BYTES of traffic run on
    // the chain word kernel when their chains are long: its small items
    // spread the pass over every SM and each thread has 64 loads in flight,
    // where the rank-streaming kernel takes one item (a chunk tile) per CTA
    // and its P tiles one after another, and the element-wise kernel folds a
    // chain in few threads.  Measured (fused ring, µs per call in a CUDA
    // graph, against the previous kernels): P = 64 at 1-64 KiB per rank
    // 5.4-5.6 against 7.2-19, 256 KiB 22.5 against 33; P = 16 at 4-64 KiB
    // 3.2-4.7 against 5.1-11.7, 1 MiB 11.1 against 18.2; P = 8 at 64 KiB-1
    // MiB 5-12% faster, at <= 16 KiB slower (the element-wise kernel's one
    // launch is near the launch floor there) and at 4 MiB (64 MiB of
    // traffic: the rank-streaming kernel fills the GPU), P = 2 slower at every
    // size; the step form's rounds (P chains of two inputs each) slower at
    // every size.
    std::vector<bool> cwords(sets.size(), false);
    for (size_t k = 0; k < sets.size(); ++k) {
        if (sets[k].empty() || S.params.form != AR_FORM_FUSED) continue;
        bool chains = true;
        int max_in = 0;
        uint64_t bytes = 0;
        for (auto& r : sets[k]) {
            const DevProg& d = lw.progs[r.prog];
            chains = chains && (d.kind == PK_CHAIN_R || d.kind == PK_CHAIN_L) && d.n_in <= kChainWordMaxIn &&
                     d.n_out <= kChainWordMaxIn;
            max_in = std::max<int>(max_in, d.n_in);
            bytes += static_cast<uint64_t>(d.n_in + b.stores(r.prog)) * (r.hi - r.lo) * es;
        }
        const bool long_chains = max_in >= 16 || (max_in >= 8 && !small[k]);
        if (chains && long_chains && bytes <= AR_CHAIN_WORD_MAX_BYTES) {
            cwords[k] = true;
            stream[k] = small[k] = false;
        }
    }
    // Fused passes whose programs all copy one input to their outputs (the
    // all-gathers) run on the copy kernel: a CTA per 16 KB item, its loads
    // in flight before its stores, where the rank-streaming kernel keeps one
    // CTA per SM and its TMA stores (90% of the copy peak against 99.5-102%;
    // the kernel has the measurements).
    std::vector<bool> copies(sets.size(), false);
    for (size_t k = 0; k < sets.size(); ++k) {
        if (sets[k].empty() || small[k] || cwords[k] || S.params.form != AR_FORM_FUSED) continue;
        bool copy = AR_COPY_KERNEL != 0;
        for (auto& r : sets[k]) {
            const DevProg& d = lw.progs[r.prog];
            copy = copy && (d.kind == PK_CHAIN_R || d.kind == PK_CHAIN_L) && d.n_in == 1 && d.n_out >= 1 &&
                   !(d.flags & PF_AVG);
        }
        if (copy) {
            copies[k] = true;
            stream[k] = false;
        }
    }
    // Fused passes of short chains or fp32 accumulations (2 ... kFewMaxIn
    // inputs: the ring's at P <= 16) run on the few-input kernel, the copy
    // kernel's grid shape (measured at 128-256 MiB per rank: see the kernel).
    // Sets of single trees (with chains) of up to kFewTreeMaxIn leaves that
    // write every rank (the allreduce's trees, not a reduce-scatter's, which
    // measured 2 points slower there) take its tree instantiation, when
    // their stacks fit the registers it keeps for them.
    std::vector<bool> few(sets.size(), false), few_trees(sets.size(), false);
    for (size_t k = 0; k < sets.size(); ++k) {
        if (sets[k].empty() || small[k] || cwords[k] || copies[k] || S.params.form != AR_FORM_FUSED) continue;
        bool flat = AR_FEW_KERNEL != 0, tree = AR_FEW_KERNEL != 0 && AR_FEW_TREES != 0, any_tree = false;
        const int stack = few_tree_stack(set_max_in(lw, sets[k]));
        // programs of more inputs than one group (the grouped variant) only
        // in sets of at least AR_FEW_LONG_MIN_BYTES: P = 64 at 4-8 MiB per
        // rank measured 78-85% of the copy peak there against 87-89% on the
        // rank-streaming kernel, at 16-256 MiB 92-98% against 86-96%
        uint64_t set_bytes = 0;
        for (auto& r : sets[k])
            set_bytes += static_cast<uint64_t>(lw.progs[r.prog].n_in + b.stores(r.prog)) * (r.hi - r.lo) * es;
        const int flat_max = AR_FEW_LONG && set_bytes >= AR_FEW_LONG_MIN_BYTES ? AR_MAX_RANKS : kFewMaxIn;
        for (auto& r : sets[k]) {
            const DevProg& d = lw.progs[r.prog];
            const bool size_ok = d.n_in >= 2 && d.n_in <= kFewMaxIn;
            const bool chain = d.kind == PK_CHAIN_R || d.kind == PK_CHAIN_L;
            flat = flat && d.n_in >= 2 && d.n_in <= flat_max && (chain || d.kind == PK_ACC);
            tree = tree && size_ok && d.n_in <= kFewTreeMaxIn &&
                   (chain || (d.kind == PK_TREE && d.n_tmp <= stack && d.n_out >= 2));
            any_tree = any_tree || d.kind == PK_TREE;
        }
        if (flat || (tree && any_tree)) {
            few[k] = true;
            few_trees[k] = !flat;
            stream[k] = false;
        }
    }
    bool stream_trees = false;
    lw.stream_slots = 0;  // shared-memory tiles for the deepest tree stack
    for (size_t k = 0; k < sets.size(); ++k)
        for (auto& r : sets[k])
            if (stream[k] && !small[k] && lw.progs[r.prog].kind == PK_TREE) {
                stream_trees = true;
                lw.stream_slots = std::max<int>(lw.stream_slots, lw.progs[r.prog].n_tmp);
            }
    // staged-kernel geometry from the programs that own an aligned body
    lw.max_in = 1;
    lw.max_tmp = 0;
    for (size_t k = 0; k < sets.size(); ++k)
        for (auto& r : sets[k]) {
            const DevProg& d = lw.progs[r.prog];
            lw.max_in_all = std::max<int>(lw.max_in_all, d.n_in);
            lw.max_tmp_all = std::max<int>(lw.max_tmp_all, d.n_tmp);
            int64_t a = (r.lo + V - 1) / V * V, e = r.hi / V * V;
            if (a < e && !stream[k] && !small[k] && !words[k] && !cwords[k] && !copies[k] && !few[k]) {
                lw.max_in = std::max<int>(lw.max_in, d.n_in);
                if (!(opt.jit_dag && AR_JIT_GEOMETRY)) lw.max_tmp = std::max<int>(lw.max_tmp, d.n_tmp);
            }
        }
    // deepest pipeline (up to kStages) that keeps tiles >= AR_MIN_TILE, else 2 stages
    int64_t t = 0;
    lw.stages = 2;
    for (int st = std::max(kStages, 2); st >= 2; --st) {
        t = (kSmemBudget - kBarrierBytes) / (st * lw.max_in + lw.max_tmp);
        lw.stages = st;
        if (t >= AR_MIN_TILE) break;
    }
    // compiled programs of 5 ... 16 inputs (the 16-byte consumers, no
    // temporaries): the depth measured best for that input count.  Forced
    // depths 2 ... 7 at 64-128 MiB per rank, fp32 and bf16, generalized and
    // RD max / min plans: against the rule above +1 point at P = 5, +2 ... +5 at
    // P = 8 and 10 ... 14 (-1.6 for bf16 RD max at P = 8), the same elsewhere.
    static const int kStagesByInputs[17] = {0, 0, 0, 0, 0, 6, 5, 5, 5, 4, 4, 4, 4, 3, 3, 2, 2};
    if (opt.jit_dag && AR_JIT_GEOMETRY && AR_JIT_STAGE_TABLE && lw.max_in >= 5 && lw.max_in <= kWordConsumerMinIn &&
        lw.max_tmp == 0)
        lw.stages = kStagesByInputs[lw.max_in];
    t = (kSmemBudget - kBarrierBytes) / (lw.stages * lw.max_in + lw.max_tmp);
    t = std::min<int64_t>(t, kMaxTileBytes);
    t = t >= 512 ? t / 512 * 512 : std::max<int64_t>(16, t / 16 * 16);
    lw.tile_bytes = static_cast<int>(t);
    // compiled programs of many inputs: tiles of 2 or 1 KB (whole words for
    // every consumer thread), the larger that keeps AR_JIT_WORD_STAGES
    // stages, with as many stages as fit (at most kStagesWord).  4 KB tiles
    // (3 stages at P = 17 / 18) measured 45% of the copy peak against 73-75%
    // with 2 KB and 6 stages (fp32 sum / max, P = 17, 64 MiB per rank).
    if (opt.jit_dag && AR_JIT_GEOMETRY && lw.max_in > kWordConsumerMinIn) {
        const int64_t room = kSmemBudget - kBarrierBytes;
        int64_t wt = kWordTileUnit;
        for (int64_t c = 2 * kWordTileUnit; c > kWordTileUnit; c /= 2)
            if (room / (c * lw.max_in) >= AR_JIT_WORD_STAGES) {
                wt = c;
                break;
            }
        lw.tile_bytes = static_cast<int>(wt);
        lw.stages = static_cast<int>(std::min<int64_t>(kStagesWord, room / (wt * lw.max_in)));
        if (lw.stages < 2) throw std::length_error("staged kernel: too many inputs per program");
    }
    // bf16 fp32 accumulation keeps 8 fp32 per 16-byte vector: 24 KB rank
    // tiles (6 vectors per thread: with 32 KB tiles the 64 accumulators and
    // the tile loads exceed the 168 registers a 320-thread CTA gets, and the
    // kernel spills; measured 24 KB with 7 stages against 32 KB with 7,
    // 24 KB with 9 and 16 KB with 14: +2-4% at P = 4 ... 64 over 32 KB, e.g.
    // P = 64 95.2% against 92.5% of the copy peak).  A tree keeps depth - 1 stack tiles in shared
    // memory next to the stages: 32 KB tiles while that leaves a pipeline of
    // at least 3 stages (trees of up to 16 leaves; measured +6% at P = 16 over
    // 16 KB tiles), 24 KB tiles for deeper trees (3 stages at 64 leaves, 4 at
    // 32; measured +7% / +12% fp32 and +10% / +11% bf16 at P = 64 / 32 over
    // 16 KB tiles with 8 / 9 stages).
    bool acc_streamed = false;
    for (size_t k = 0; k < sets.size(); ++k)
        if (stream[k] && !small[k])
            for (auto& r : sets[k]) acc_streamed |= lw.progs[r.prog].kind == PK_ACC;
    const bool bf16_acc = S.dtype == AR_BFLOAT16 && acc_streamed;
    const bool deep = stream_trees && lw.stream_slots > AR_TREE_WIDE_SLOTS;
    lw.stream_trees = stream_trees;
    // deep trees: the stack in tensor memory, so 32 KB tiles and shared
    // memory for stages only.  Measured at 64 MiB per rank against the
    // shared-memory stack (24 KB tiles, 3 stages): P = 64 RH / binomial fp32
    // 88% -> 95-96%, bf16 86% -> 94%, int32 88% -> 95%, the RH reduce-scatter
    // 80% -> 98%; P = 32 90% -> 94-95%; 4 stages against 5 and 7 +1-2%.
    // From 4 stack entries (P = 16: bf16 94% -> 96%, fp32 equal); at 3 (P = 8)
    // the shared-memory stack's pipeline measured 1.7% faster.
    lw.stream_tmem = stream_trees && AR_TMEM_TREES && lw.stream_slots > AR_TMEM_TREE_MIN_SLOTS && lw.stream_slots <= 8;
    lw.stream_tile = bf16_acc ? AR_BF16_ACC_TILE : (deep && !lw.stream_tmem) ? kStreamTileTree : kStreamTileBytes;
    lw.stream_stages = std::min(kMaxStages, (kStreamSmemBudget - kBarrierBytes) / lw.stream_tile -
                                                (lw.stream_tmem ? 0 : lw.stream_slots));
    if (lw.stream_tmem) lw.stream_stages = std::min(lw.stream_stages, AR_TMEM_TREE_STAGES);
    // Chains over 4-byte elements stream best with a short pipeline: with 7
    // stages in flight per SM the reads crowd out the writes.  Measured at
    // 256 MiB per rank, 3 stages against 7: fused ring +4% at P = 4 and 8,
    // +7% at P = 6, within 2% either way at P = 2, 12 ... 64; the step rounds
    // of every schedule at P = 8 up to +2%.  fp32 accumulation (fp32 and
    // int32 elements) peaks at 5 stages: +4% over 7 at P = 8, equal at 64.
    // bf16 chains, one bf16x2 instruction (or compare) per element pair,
    // peak at 4: against 7, sum fused ring +1% at P = 8, +3% at P = 16 and
    // 64, step rounds +1%, the reduce-scatter +5%; max / min +3-4%.  bf16
    // fp32 accumulation on 24 KB tiles: 7 stages (9 fit) measured +2-3% at
    // P = 4 ... 16, within 1% at 32 and 64.
    if (!stream_trees && es == 4)
        lw.stream_stages = std::min(lw.stream_stages, acc_streamed ? AR_ACC_STAGES_4B : AR_CHAIN_STAGES_4B);
    if (!stream_trees && es == 2 && !acc_streamed) lw.stream_stages = std::min(lw.stream_stages, AR_CHAIN_STAGES_BF16);
    if (!stream_trees && es == 2 && acc_streamed) lw.stream_stages = std::min(lw.stream_stages, AR_ACC_STAGES_BF16);
    // The TMA-store epilogue holds an item's last stage until its outputs are
    // copied out.  Measured at the bench size with the pipelines above: in a
    // fused pass it wins for copies (one input, many outputs: the all-gather,
    // +2%), for few inputs and outputs (P = 2, bf16 +3%) and for bf16 fp32
    // accumulation, whose direct stores are costly (+30%); 128-bit stores
    // from registers win with many outputs (allreduce at P >= 8, up to +5%)
    // and with many inputs per output (the reduce-scatter: bf16 ring +4%, RH
    // +1%).  The step form's rounds run faster with 128-bit stores in every
    // round, copies included: ring, pipeline, binomial, generalized at P = 8
    // and 12 +1-3.5% over TMA stores (and over TMA stores in either kind of
    // round alone) — except bf16 rounds whose transfers have two outputs
    // (recursive doubling's exchanges: TMA stores +3.5%, as for P = 2).
    const bool rounds = sets.size() > 1 || S.params.form == AR_FORM_STEP;
    auto tma_store = [&](const std::vector<Range>& set) {
        if (S.dtype == AR_BFLOAT16 && acc_streamed) return AR_BF16_ACC_TMA != 0;
        int max_out = 0, max_in = 0;
        for (auto& r : set) {
            max_out = std::max<int>(max_out, lw.progs[r.prog].n_out);
            max_in = std::max<int>(max_in, lw.progs[r.prog].n_in);
        }
        const bool few = max_out <= AR_TMA_STORE_MAX_OUT && max_in <= 4;
        if (rounds) return S.dtype == AR_BFLOAT16 && few && max_out >= 2;
        return max_in <= 1 || few;
    };
    for (size_t k = 0; k < sets.size(); ++k) {
        LaunchSet ls;
        ls.stream = stream[k];
        ls.tma_store = stream[k] && tma_store(sets[k]);
        int64_t tile_bytes = cwords[k]   ? chain_word_item_bytes(set_max_in(lw, sets[k]))
                             : copies[k] || few[k] ? kCopyItemBytes
                             : words[k]  ? kWordItemBytes
                             : stream[k] ? lw.stream_tile
                                         : lw.tile_bytes;
        if (cwords[k]) {
            // a small pass: items of down to 512 B so that there are about two
            // per SM (each thread then has fewer positions, but the pass runs
            // on more SMs at once)
            int64_t rank_bytes = 0;
            for (auto& r : sets[k]) rank_bytes += (r.hi - r.lo) * es;
            const int64_t want = (rank_bytes / (2 * kSpreadItems) + 511) / 512 * 512;
            tile_bytes = std::max<int64_t>(4 * kChainWordThreads, std::min(tile_bytes, want));
        }
        const int64_t tile_elems = item_elems(sets[k], tile_bytes / es, V);
        for (auto& r : sets[k]) {
            int64_t a = (r.lo + V - 1) / V * V, e = r.hi / V * V;
            if (a < e) {
                if (r.lo < a) ls.edge.push_back({r.lo, static_cast<uint32_t>(a - r.lo), r.prog});
                for (int64_t x = a; x < e; x += tile_elems)
                    ls.bulk.push_back({x, static_cast<uint32_t>(std::min(tile_elems, e - x)), r.prog});
                if (e < r.hi) ls.edge.push_back({e, static_cast<uint32_t>(r.hi - e), r.prog});
            } else {
                ls.edge.push_back({r.lo, static_cast<uint32_t>(r.hi - r.lo), r.prog});
            }
            // element-wise items: one block of the element kernel each for a
            // small set (parallelism), 4096 elements otherwise
            const int64_t fb = small[k] ? kElemBlock : 4096;
            for (int64_t x = r.lo; x < r.hi; x += fb)
                ls.fallback.push_back({x, static_cast<uint32_t>(std::min<int64_t>(fb, r.hi - x)), r.prog});
            const DevProg& d = lw.progs[r.prog];
            ls.bytes += static_cast<uint64_t>(d.n_in + b.stores(r.prog)) * (r.hi - r.lo) * es;
        }
        ls.small = small[k];
        ls.words = words[k];
        ls.chain_words = cwords[k];
        ls.copies = copies[k];
        ls.few = few[k];
        ls.few_trees = few_trees[k];
        ls.max_in = set_max_in(lw, sets[k]);
        ls.chains = !sets[k].empty();
        for (auto& r : sets[k]) {
            const DevProg& d = lw.progs[r.prog];
            ls.chains = ls.chains && (d.kind == PK_CHAIN_R || d.kind == PK_CHAIN_L) && d.n_in <= kChainWordMaxIn &&
                        d.n_out <= kChainWordMaxIn;
        }
        lw.hbm_bytes += ls.bytes;
        lw.n_items += ls.small ? ls.fallback.size() : ls.bulk.size() + ls.edge.size();
        lw.launches += ls.small ? 1 : (!ls.bulk.empty()) + (!ls.edge.empty());
        lw.sets.push_back(std::move(ls));
    }
}

std::vector<Window> host_windows(const LaunchSet& ls, int64_t n, uint64_t total_bytes) {
    std::vector<Window> out;
    const size_t nb = ls.bulk.size(), ne = ls.edge.size();
    const uint64_t W = std::min<uint64_t>({total_bytes / (128ull << 20), 32, static_cast<uint64_t>(nb)});
    if (W < 2) return out;
    // suffix_lo[b]: the lowest start of items b.., prefix_hi: the highest end of items ..b-1
    std::vector<int64_t> suffix_lo(nb + 1, n);
    for (size_t b = nb; b-- > 0;) suffix_lo[b] = std::min(suffix_lo[b + 1], ls.bulk[b].elem);
    std::vector<size_t> cuts(1, 0);
    int64_t prefix_hi = 0;
    size_t best = 0;  // the last valid cut seen
    uint64_t w = 1;
    for (size_t b = 0; b < nb && w < W; ++b) {
        if (b > 0 && prefix_hi <= suffix_lo[b]) best = b;
        while (w < W && b >= nb * w / W) {  // cut w is due at item nb w / W: take the last valid one
            if (best > cuts.back()) cuts.push_back(best);
            ++w;
        }
        prefix_hi = std::max(prefix_hi, ls.bulk[b].elem + static_cast<int64_t>(ls.bulk[b].count));
    }
    if (cuts.size() < 2) return out;
    cuts.push_back(nb);
    auto first_edge_at = [&](int64_t x) {
        uint32_t k = 0;
        while (k < ne && ls.edge[k].elem < x) ++k;
        return k;
    };
    for (size_t k = 0; k + 1 < cuts.size(); ++k) {
        Window win;
        win.b0 = static_cast<uint32_t>(cuts[k]);
        win.b1 = static_cast<uint32_t>(cuts[k + 1]);
        win.lo = k == 0 ? 0 : suffix_lo[cuts[k]];
        win.hi = k + 2 == cuts.size() ? n : suffix_lo[cuts[k + 1]];
        win.e0 = k == 0 ? 0 : first_edge_at(win.lo);
        win.e1 = k + 2 == cuts.size() ? static_cast<uint32_t>(ne) : first_edge_at(win.hi);
        out.push_back(win);
    }
    // check: consecutive windows over [0, n), every item inside its window
    bool ok = out.front().lo == 0 && out.back().hi == n && out.back().b1 == nb && out.back().e1 == ne;
    for (size_t k = 0; k < out.size() && ok; ++k) {
        const Window& x = out[k];
        ok = x.lo < x.hi && x.b0 < x.b1 && x.e0 <= x.e1 && x.hi <= n &&
             (k == 0 || (x.lo == out[k - 1].hi && x.b0 == out[k - 1].b1 && x.e0 == out[k - 1].e1));
        for (uint32_t b = x.b0; b < x.b1 && ok; ++b)
            ok = ls.bulk[b].elem >= x.lo && ls.bulk[b].elem + static_cast<int64_t>(ls.bulk[b].count) <= x.hi;
        for (uint32_t b = x.e0; b < x.e1 && ok; ++b)
            ok = ls.edge[b].elem >= x.lo && ls.edge[b].elem + static_cast<int64_t>(ls.edge[b].count) <= x.hi;
    }
    if (!ok) out.clear();
    return out;
}

LoweringCheck check_lowering(const Lowered& L, int64_t n, int es, const std::vector<Window>& windows) {
    LoweringCheck c;
    using Span = std::pair<int64_t, int64_t>;
    // sorted, merged spans; {-1, -1} marks an overlap
    auto merged = [](std::vector<Span> v) {
        std::sort(v.begin(), v.end());
        std::vector<Span> m;
        for (const Span& x : v) {
            if (!m.empty() && m.back().second > x.first) return std::vector<Span>{{-1, -1}};
            if (!m.empty() && m.back().second == x.first)
                m.back().second = x.second;
            else
                m.push_back(x);
        }
        return m;
    };
    for (const LaunchSet& ls : L.sets) {
        std::map<uint32_t, std::vector<Span>> want, got;
        for (const WorkItem& w : ls.fallback) want[w.prog].push_back({w.elem, w.elem + w.count});
        for (const WorkItem& w : ls.bulk) {
            got[w.prog].push_back({w.elem, w.elem + w.count});
            if (w.count == 0 || (w.elem * es) % 16 || (static_cast<int64_t>(w.count) * es) % 16) c.tiling_ok = false;
        }
        for (const WorkItem& w : ls.edge) got[w.prog].push_back({w.elem, w.elem + w.count});
        c.items += ls.bulk.size() + ls.edge.size();
        if (want.size() != got.size()) c.tiling_ok = false;
        for (auto& kv : want) {
            auto g = got.find(kv.first);
            if (g == got.end() || merged(kv.second) != merged(g->second)) c.tiling_ok = false;
        }
        if (ls.stream && !ls.small && !ls.bulk.empty()) {
            const size_t G = std::min<size_t>(152, ls.bulk.size());
            std::vector<double> share(G, 0.0);
            double total = 0;
            for (size_t i = 0; i < ls.bulk.size(); ++i) {
                const DevProg& d = L.progs[ls.bulk[i].prog];
                const double b = static_cast<double>(d.n_in + d.n_out) * ls.bulk[i].count;
                share[i % G] += b;
                total += b;
            }
            c.wave_balance = std::max(c.wave_balance, *std::max_element(share.begin(), share.end()) / (total / G));
        }
    }
    if (!windows.empty()) {
        const LaunchSet& ls = L.sets.at(0);
        std::vector<int> bulk_seen(ls.bulk.size(), 0), edge_seen(ls.edge.size(), 0);
        int64_t at = 0;
        for (const Window& w : windows) {
            if (w.lo != at || w.hi <= w.lo || w.hi > n || w.b1 > ls.bulk.size() || w.e1 > ls.edge.size()) {
                c.windows_ok = false;
                break;
            }
            at = w.hi;
            for (uint32_t b = w.b0; b < w.b1; ++b) {
                ++bulk_seen[b];
                if (ls.bulk[b].elem < w.lo || ls.bulk[b].elem + ls.bulk[b].count > w.hi) c.windows_ok = false;
            }
            for (uint32_t b = w.e0; b < w.e1; ++b) {
                ++edge_seen[b];
                if (ls.edge[b].elem < w.lo || ls.edge[b].elem + ls.edge[b].count > w.hi) c.windows_ok = false;
            }
        }
        if (at != n) c.windows_ok = false;
        for (int x : bulk_seen) c.windows_ok &= x == 1;
        for (int x : edge_seen) c.windows_ok &= x == 1;
    }
    return c;
}

}  // namespace ar
