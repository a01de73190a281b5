// Lowering of a compiled schedule to tile programs and work items.
#pragma once

#include <cstdint>
#include <vector>

#include "devprog.hpp"
#include "schedule.hpp"

namespace ar {

// One kernel-launch set: the items of one fused pass or of one round.
struct LaunchSet {
    std::vector<WorkItem> bulk;      // 16-byte aligned ranges, staged kernel
    std::vector<WorkItem> edge;      // unaligned heads / tails, element kernel
    std::vector<WorkItem> fallback;  // whole ranges for unaligned buffers
    uint64_t bytes = 0;              // algorithmic HBM bytes of the set
};

struct Lowered {
    std::vector<DevProg> progs;
    std::vector<uint16_t> refs;
    std::vector<uint32_t> ins;
    std::vector<LaunchSet> sets;
    int tile_bytes = 0;   // bytes per input tile of the staged kernel
    int stages = 0;       // pipeline depth of the staged kernel
    int max_in = 0;       // largest n_in of a program used by bulk items
    int max_tmp = 0;      // largest n_tmp of such a program
    int max_in_all = 0;   // largest n_in / n_tmp over all programs
    int max_tmp_all = 0;
    uint64_t hbm_bytes = 0;
    uint64_t n_items = 0;
    int launches = 0;     // launches per execute on aligned buffers
};

// Staged-kernel shared-memory budget (bytes) shared by lowering and launch.
constexpr int kSmemBudget = 200 * 1024;
constexpr int kMaxTileBytes = 32 * 1024;
constexpr int kStages = 3;

// Builds the fused pass (one set) or the rounds (one set per round).
void lower(const Schedule& S, Lowered& out);

// Dynamic shared memory the staged kernel needs for a lowering.
int staged_smem_bytes(const Lowered& lw);

}  // namespace ar
