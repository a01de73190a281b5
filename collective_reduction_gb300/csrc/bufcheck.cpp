// Rank-buffer checks shared by every entry point that launches kernels on
// caller memory.  The C ABI promises AR_ERR_INVALID_ARG, not a fault, for a
// pointer that is not device memory of the current device (pageable or
// pinned host memory, another GPU's memory) or whose n elements run past the
// allocation holding it: both are caught here, before any launch.
#include "bufcheck.hpp"

#include <cuda.h>  // CUresult / CUdeviceptr only: the driver call is resolved at run time
#include <cuda_runtime.h>

#include <algorithm>
#include <utility>
#include <vector>

namespace ar {
namespace {

using AddressRangeFn = CUresult (*)(CUdeviceptr*, size_t*, CUdeviceptr);

// cuMemGetAddressRange through the runtime's driver entry-point query (the
// library links only the static runtime); null if the driver has none.
AddressRangeFn address_range() {
    static const AddressRangeFn fn = [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuMemGetAddressRange", &f, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess) {
            cudaGetLastError();
            return static_cast<AddressRangeFn>(nullptr);
        }
        return reinterpret_cast<AddressRangeFn>(f);
    }();
    return fn;
}

// Device (or managed) memory of `device`, with `bytes` inside its allocation.
bool resident(const void* p, uint64_t bytes, int device) {
    cudaPointerAttributes at{};
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
        cudaGetLastError();  // an unknown pointer is the caller's error, not a sticky one
        return false;
    }
    if (at.type == cudaMemoryTypeDevice) {
        if (at.device != device) return false;
    } else if (at.type != cudaMemoryTypeManaged) {
        return false;  // unregistered (pageable) or pinned host memory
    }
    if (AddressRangeFn range = address_range()) {
        CUdeviceptr base = 0;
        size_t size = 0;
        const CUdeviceptr a = reinterpret_cast<CUdeviceptr>(p);
        if (range(&base, &size, a) == CUDA_SUCCESS) {
            if (a < base || a - base > size || bytes > size - (a - base)) return false;
        }
    }
    return true;
}

}  // namespace

ar_status check_rank_buffers(int P, uint64_t n, int es, int device, void* const* bufs, bool residency,
                             bool* aligned16) {
    if (!bufs || P < 1 || es < 1) return AR_ERR_INVALID_ARG;
    const uint64_t bytes = n * static_cast<uint64_t>(es);
    std::vector<std::pair<uintptr_t, int>> addr;
    addr.reserve(P);
    bool aligned = true;
    for (int r = 0; r < P; ++r) {
        const uintptr_t a = reinterpret_cast<uintptr_t>(bufs[r]);
        if (!a || a % es) return AR_ERR_INVALID_ARG;
        if (a + bytes < a) return AR_ERR_INVALID_ARG;  // the range wraps the address space
        aligned = aligned && a % 16 == 0;
        addr.emplace_back(a, r);
    }
    std::sort(addr.begin(), addr.end());
    for (int r = 0; r + 1 < P; ++r)
        if (addr[r].first == addr[r + 1].first || addr[r].first + bytes > addr[r + 1].first) return AR_ERR_INVALID_ARG;
    if (residency)
        for (int r = 0; r < P; ++r)
            if (!resident(bufs[r], bytes, device)) return AR_ERR_INVALID_ARG;
    if (aligned16) *aligned16 = aligned;
    return AR_OK;
}

}  // namespace ar
