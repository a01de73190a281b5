// Lowering of a compiled schedule to tile programs and work items.
#pragma once

#include <algorithm>
#include <cstdint>
#include <vector>

#include "devprog.hpp"
#include "schedule.hpp"

namespace ar {

// One kernel-launch set: the items of one fused pass or of one round.
struct LaunchSet {
    std::vector<WorkItem> bulk;      // 16-byte aligned ranges: rank-streaming or staged kernel
    std::vector<WorkItem> edge;      // unaligned heads / tails, element kernel
    std::vector<WorkItem> fallback;  // whole ranges for unaligned buffers
    uint64_t bytes = 0;              // algorithmic HBM bytes of the set
    bool stream = false;             // bulk items run on the rank-streaming kernel
    bool tma_store = false;          // ... with the TMA bulk-store epilogue (else 128-bit stores)
    bool small = false;              // small set (<= 256 KB): one element-wise launch over fallback
    bool words = false;              // bulk items run on the run-time compiled word kernel
    bool chain_words = false;        // bulk items run on the chain word kernel
    bool copies = false;             // bulk items run on the copy kernel (one input, many outputs)
    bool few = false;                // bulk items run on the few-input kernel
    bool few_trees = false;          // ... its instantiation for single trees (and chains)
    int max_in = 0;                  // most inputs of a program of the set
    bool chains = false;             // every program is a chain the chain word kernel runs
};

struct Lowered {
    std::vector<DevProg> progs;
    std::vector<uint16_t> refs;
    std::vector<uint32_t> ins;
    std::vector<LaunchSet> sets;
    int tile_bytes = 0;   // bytes per input tile of the staged kernel
    int stages = 0;       // pipeline depth of the staged kernel
    int stream_tile = 0;  // bytes per rank tile of the rank-streaming kernel
    int stream_stages = 0;
    bool stream_trees = false;      // rank-streaming kernel: the instantiation that runs TREE programs
    bool stream_tmem = false;       // ... with the tree stack in tensor memory (no stack tiles)
    int stream_slots = 0;           // rank-streaming kernel: shared-memory tiles of the tree stack
    int max_in = 0;       // largest n_in of a program used by bulk items
    int max_tmp = 0;      // largest n_tmp of such a program
    int max_in_all = 0;   // largest n_in / n_tmp over all programs
    int max_tmp_all = 0;
    uint64_t hbm_bytes = 0;
    uint64_t n_items = 0;
    int launches = 0;     // launches per execute on aligned buffers
    int phys_slots = 1;   // step form: physical copies per rank buffer (slots and their twins)
};

// Staged-kernel geometry shared by lowering and launch: shared-memory budget
// per CTA (the GB300 opt-in maximum), largest input tile, pipeline depth
// (the deepest up to AR_STAGES whose tiles stay >= 6 KB).  Measured on the
// run-time compiled DAG kernels at 256 MiB per rank: 4 stages in 227 KB
// against 3 in 200 KB, P = 7 generalized r = 1 / r = 3 +3% / +4% fp32, r = 1
// bf16 and RD max bf16 at P = 8 +2%; 5 stages against 4 (P <= 7 only: 6 KB
// tiles) +3-4 points of the copy peak at P = 6 and 7, +0.5 at P = 5.  Deeper
// pipelines of 4-5 KB tiles measured -12 ... +7 points plan by plan (P = 5 ...
// 16) and are not taken.
#ifndef AR_SMEM_BUDGET
#define AR_SMEM_BUDGET (227 * 1024)
#endif
#ifndef AR_MAX_TILE
#define AR_MAX_TILE kMaxStagedTile
#endif
#ifndef AR_STAGES
#define AR_STAGES 5
#endif
constexpr int kSmemBudget = AR_SMEM_BUDGET;
constexpr int kMaxTileBytes = AR_MAX_TILE;
constexpr int kStages = AR_STAGES;        // staged kernel: preferred pipeline depth
// the rank-streaming kernel keeps no temporaries: its stages may use the
// whole opt-in shared memory of a GB300 SM (227 KB)
constexpr int kStreamSmemBudget = 227 * 1024;
static_assert(kMaxTileBytes <= kMaxStagedTile, "staged tiles beyond what the consumers cover");
// full, empty and ready barriers (8 bytes each) per stage in the barrier area
constexpr int kMaxStages = kBarrierBytes / 24;

// The word kernel (run-time compiled): one thread per 32-bit word of every
// rank, threads per CTA, rank bytes per work item, and its prefetch depth:
// stages of kWordThreads words of every input in shared memory (as many as
// fit in about 220 KB, at most 4).
constexpr int kWordThreads = 256;
constexpr int kWordItemBytes = 32768;
inline int word_kernel_stages(int max_in) {
    const int fit = (220 * 1024) / (4 * kWordThreads * std::max(max_in, 1));
    return std::min(4, fit);
}
inline int word_kernel_smem(int max_in) { return word_kernel_stages(max_in) * max_in * 4 * kWordThreads; }
// The copy kernel: rank bytes per work item (one item per CTA).
#ifndef AR_COPY_ITEM_BYTES
#define AR_COPY_ITEM_BYTES 16384
#endif
constexpr int kCopyItemBytes = AR_COPY_ITEM_BYTES;
// The chain word kernel: rank bytes per work item for programs of n_in
// inputs (one round of its threads: kChainWordMaxIn / n_in words each), and
// the largest set (bytes of traffic) it takes.
inline int chain_word_item_bytes(int n_in) {
    return 4 * kChainWordThreads * (n_in <= 8 ? 8 : n_in <= 16 ? 4 : 1);
}
#ifndef AR_CHAIN_WORD_MAX_BYTES
#define AR_CHAIN_WORD_MAX_BYTES (32ull << 20)
#endif

struct LowerOptions {
    // The staged launches' DAG programs will run as run-time compiled code:
    // the staged kernel's geometry then reserves no shared-memory
    // temporaries (the interpreter's), and programs of many inputs get
    // tiles of whole 1 KB units (their compiled consumers take one 32-bit
    // word per thread).
    bool jit_dag = false;
    // Sets with DAG programs of at least word_min_in inputs and at least
    // word_min_bytes of traffic run on the word kernel (needs the run-time
    // compiler); the others on the staged kernel.
    bool word_dag = false;
    int word_min_in = 1;
    uint64_t word_min_bytes = 0;
};

// Compiled staged consumers take one 32-bit word of every input per thread
// (rather than 16-byte vectors) for programs of more than this many inputs.
constexpr int kWordConsumerMinIn = 16;
constexpr int kWordTileUnit = 4 * 32 * kConsumerWarps;  // one word per consumer thread

// Builds the fused pass (one set) or the rounds (one set per round).
void lower(const Schedule& S, Lowered& out, const LowerOptions& opt = LowerOptions());

// Element window of a fused pass for the pipelined host path: elements
// [lo, hi) of every rank, bulk items [b0, b1) and edge items [e0, e1).
struct Window {
    int64_t lo, hi;
    uint32_t b0, b1, e0, e1;
};

// About 128 MB of rank data per window, at most 32 windows, consecutive and
// covering [0, n).  A window ends only between bulk items b - 1 and b where
// every item before b ends at or before the start of every item from b on,
// so each window's items lie inside its elements whatever the order of the
// item list.  Every window is checked against the items before it is
// returned; on any mismatch the result is empty and the host path runs as
// one pass (a window's copies must never leave the rank buffers).
std::vector<Window> host_windows(const LaunchSet& ls, int64_t n, uint64_t total_bytes);

// Checks of a lowering that share no code with it: whether the bulk and edge
// items of every set tile its ranges (taken from the set's whole-range
// fallback items) program by program, bulk items 16-byte aligned; whether
// the windows are consecutive over [0, n) with every item inside its
// window; and the round-robin byte balance of the streamed sets over 152
// CTAs (largest share / mean share).
struct LoweringCheck {
    bool tiling_ok = true;
    bool windows_ok = true;
    double wave_balance = 1.0;
    uint64_t items = 0;
};
LoweringCheck check_lowering(const Lowered& L, int64_t n, int es, const std::vector<Window>& windows);

// Dynamic shared memory the staged / rank-streaming kernels need.
int staged_smem_bytes(const Lowered& lw);
int stream_smem_bytes(const Lowered& lw);

}  // namespace ar
