// Checks of the caller's rank buffers before any kernel may touch them, and
// the trace range every launching entry point opens.
#pragma once

#include <nvtx3/nvToolsExt.h>

#include <cstdint>

#include "ar.h"

namespace ar {

// An NVTX range over one C-ABI call, seen by profilers that attach an NVTX
// tool (a no-op function call otherwise).
struct TraceRange {
    explicit TraceRange(const char* name) { nvtxRangePushA(name); }
    ~TraceRange() { nvtxRangePop(); }
    TraceRange(const TraceRange&) = delete;
    TraceRange& operator=(const TraceRange&) = delete;
};

// P pointers to n elements of es bytes each.  Always checked: non-null,
// aligned to the element size, pairwise disjoint address ranges.  With
// `residency` also: each pointer is device memory of `device` (or managed
// memory) according to cudaPointerGetAttributes, and its n elements lie
// inside the allocation that holds it (cuMemGetAddressRange; skipped where the
// driver cannot report the range).  Launches nothing.  *aligned16 is set when
// every pointer is 16-byte aligned.  AR_ERR_INVALID_ARG on any failure.
ar_status check_rank_buffers(int P, uint64_t n, int es, int device, void* const* bufs, bool residency,
                             bool* aligned16);

}  // namespace ar
