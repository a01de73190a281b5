// Launch arguments and status bits shared by the compiled kernels, the
// run-time compiled DAG kernels and the host code that launches them.
#pragma once

#if !defined(__CUDACC_RTC__)
#include <cstdint>
#endif

#include "ar.h"
#include "devprog.hpp"

namespace ar {

// Everything a launch needs, passed by value (fits the kernel parameter space).
struct KernelArgs {
    void* bufs[AR_MAX_RANKS];  // slot-0 buffers, one per rank
    char* scratch;             // slots >= 1
    uint64_t slot_stride;      // bytes between scratch buffers
    const WorkItem* items;
    const DevProg* progs;
    const uint16_t* refs;
    const uint32_t* ins;
    int* status;               // device status word (bit flags, 0 = fine)
    uint32_t n_items;
    int P;
    int tile_bytes;            // staged kernel: bytes per input tile
    int stages;                // staged kernel: pipeline depth
    int max_in;                // staged: input tiles per stage; element kernel: value rows
    int max_tmp;               // staged: temporary tiles; element kernel: temp rows
    int flags;                 // kArg* bits
};

// KernelArgs::flags: the rank-streaming kernel writes results back to shared
// memory and copies them out with TMA bulk stores (else 128-bit stores)
constexpr int kArgTmaStore = 1;
// KernelArgs::flags: the launch has single-tree programs (the rank-streaming
// kernel's tree instantiations; a.max_tmp stack tiles follow the stages)
constexpr int kArgTrees = 2;
// KernelArgs::flags: the tree stack lives in tensor memory (the 32 KB-tile
// tree instantiation that allocates it; a.max_tmp entries, at most 8)
constexpr int kArgTmemStack = 4;

// Status word bits written by the kernels.
constexpr int kStatusWaitFull = 1;   // a consumer gave up waiting for a stage
constexpr int kStatusWaitEmpty = 2;  // the producer gave up waiting for a free stage
constexpr int kStatusDrain = 4;      // a failing producer gave up draining its copies
constexpr int kStatusBadProgram = 8; // a program kind the launched kernel does not run

constexpr int kStagedThreads = 32 * (1 + kConsumerWarps);
constexpr int kElemThreads = kElemBlock;

}  // namespace ar
