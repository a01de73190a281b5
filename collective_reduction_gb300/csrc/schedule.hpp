// Host-side schedule compiler: turns an allreduce schedule into rounds of
// transfers and into the reduction tree every element of every rank ends with.
#pragma once

#include <cstdint>
#include <string>
#include <unordered_map>
#include <vector>

#include "ar.h"

namespace ar {

// One transfer of a round: dst_out = dst_in (+) src (combine, receiver on the
// left) or dst_out = src (copy), over elements [lo, hi) of both ranks.  Slots
// name the storage a rank uses for a chunk: slot 0 is the rank's own buffer,
// slot k >= 1 a scratch copy holding a second partial of the same chunk.
struct Transfer {
    int src, src_slot;
    int dst, dst_in, dst_out;
    int64_t lo, hi;
    bool combine;
    // AR_AVG: per segment the transfer covers (from the first), whether its
    // combine completes the reduction (that result is divided by P)
    std::vector<uint8_t> completes;
};

struct Round {
    std::vector<Transfer> xfers;
    std::vector<int64_t> sent;  // elements each rank sends (one per message)
};

// Hash-consed reduction DAG over ranks: node i < P is rank i's contribution,
// node i >= P is (left (+) right).
class Dag {
public:
    explicit Dag(int P = 0) : P_(P) {}
    int P() const { return P_; }
    bool leaf(int32_t x) const { return x < P_; }
    int32_t left(int32_t x) const { return kids_[2 * (x - P_)]; }
    int32_t right(int32_t x) const { return kids_[2 * (x - P_) + 1]; }
    int32_t combine(int32_t l, int32_t r);
    int32_t size() const { return P_ + static_cast<int32_t>(kids_.size() / 2); }
    std::string text(int32_t x) const;
    // True when node x contains every leaf exactly once.
    bool complete(int32_t x) const;

private:
    int P_;
    std::vector<int32_t> kids_;
    std::unordered_map<uint64_t, int32_t> memo_;
};

struct Params {
    int form = AR_FORM_FUSED;
    int order = AR_ORDER_FAITHFUL;
    int group = AR_GROUP_CYCLIC;
    int r = 0;
    int k1 = 0;
    std::vector<int> group_sizes;
    int blocks = 1;
    int phase = AR_PHASE_ALLREDUCE;
    int jit = AR_JIT_AUTO;
};

struct Schedule {
    int P = 0;
    int64_t n = 0;
    int dtype = 0, op = 0, algo = 0;
    Params params;
    std::vector<Round> rounds;
    int max_slots = 1;
    int64_t combines = 0;
    // Symbolic result: segment boundaries (bounds[0] = 0, bounds.back() = n),
    // and the DAG node each rank holds in slot 0 of each segment at the end.
    std::vector<int64_t> bounds;
    Dag dag;
    std::vector<int32_t> final_node;  // [rank * nseg + seg]
    // Whether the schedule defines rank's result in a segment: every rank for
    // an allreduce; the owners (complete trees) after a reduce-scatter; the
    // ranks that receive a copy in an all-gather.
    std::vector<char> defined;        // [rank * nseg + seg]
    int nseg() const { return static_cast<int>(bounds.size()) - 1; }
    int32_t final_at(int rank, int seg) const { return final_node[rank * nseg() + seg]; }
    bool defined_at(int rank, int seg) const { return defined[rank * nseg() + seg] != 0; }
    int seg_of(int64_t elem) const;  // segment containing elem (elem < n)
};

std::vector<std::pair<int64_t, int64_t>> ceil_split(int64_t n, int64_t N);
int ceil_log2(int64_t P);
int esize_of(int dtype);

// Validates the request, generates the rounds and runs them symbolically.
ar_status compile_schedule(int P, int64_t n, int dtype, int op, int algo, const ar_params* p,
                           Schedule& out);

}  // namespace ar
