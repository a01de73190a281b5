// ar_allreduce_static: the allreduce for callers that must not allocate
// device memory.
//
// Who needs it: code that runs where a cudaMalloc is unavailable or unwanted —
// a process whose device memory is entirely reserved up front by another
// allocator (a framework's caching pool that owns the GPU), a service with a
// hard device-memory budget fixed at start-up, or a latency-critical path that
// cannot afford cudaMalloc / cudaFree's implicit device-wide synchronisation.
// Such callers cannot build a plan (ar_plan_create allocates the plan's device
// tables, status word and scratch), so this entry point compiles the schedule
// on the host and runs the same kernels with all of that scratch placed in one
// file-scope static device array instead.
//
// The array is created when the CUDA module of this file is loaded on a
// device and lives until the process exits (every GPU that loads the library
// holds AR_STATIC_SCRATCH_BYTES of it).  Host code only ever sees the array's
// name as a host-side stand-in; its device address is obtained once per
// device with cudaGetSymbolAddress, on the first call made with that device
// current, and kept for the life of the process (a cudaDeviceReset after that
// call is not supported: the array may then sit elsewhere).
//
// The kernels report a bounded wait that gave up, or a program they do not
// run, in the array's status word.  ar_allreduce_static clears it at the
// start of every call; ar_allreduce_static_check reads it back.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstring>
#include <mutex>
#include <new>
#include <stdexcept>
#include <vector>

#include "ar.h"
#include "bufcheck.hpp"
#include "kargs.hpp"
#include "kernels.hpp"
#include "lower.hpp"
#include "schedule.hpp"

namespace {

// Layout of the static array: status word, tile-program tables, partial slots.
constexpr size_t kStatusArea = 256;
constexpr size_t kTableArea = AR_STATIC_TABLE_BYTES;
constexpr size_t kSlotArea = AR_STATIC_SCRATCH_BYTES - kStatusArea - kTableArea;
static_assert(AR_STATIC_SCRATCH_BYTES > kStatusArea + kTableArea, "static scratch too small");

__device__ __align__(256) unsigned char g_static_scratch[AR_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;

struct DeviceState {
    bool ready = false;
    char* base = nullptr;  // device address of g_static_scratch on this device
    int num_sms = 0;
    int optin = 0;
};

DeviceState g_dev[kMaxDevices];
std::mutex g_setup_mutex;

// First call on a device: resolve the array's device address (with that
// device current) and read the launch limits.
ar_status setup(int dev, DeviceState*& out) {
    if (dev < 0 || dev >= kMaxDevices) return AR_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    DeviceState& d = g_dev[dev];
    if (!d.ready) {
        void* p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_static_scratch);
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev);
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&d.optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
        if (e != cudaSuccess) return AR_ERR_CUDA;
        d.base = static_cast<char*>(p);
        d.ready = true;
    }
    out = &d;
    return AR_OK;
}

template <class T>
size_t put(std::vector<char>& blob, const std::vector<T>& v) {
    size_t off = (blob.size() + 255) / 256 * 256;
    blob.resize(off + v.size() * sizeof(T));
    if (!v.empty()) std::memcpy(blob.data() + off, v.data(), v.size() * sizeof(T));
    return off;
}

}  // namespace

extern "C" ar_status ar_allreduce_static(int P, uint64_t n, ar_dtype dtype, ar_op op, ar_algo algo,
                                         const ar_params* params, void* const* rank_bufs, void* stream) {
    ar::TraceRange trace("ar_allreduce_static");
    if (!rank_bufs) return AR_ERR_INVALID_ARG;
    if (n > (uint64_t(1) << 40)) return AR_ERR_UNSUPPORTED;
    try {
        ar::Schedule S;
        ar_status st = ar::compile_schedule(P, static_cast<int64_t>(n), dtype, op, algo, params, S);
        if (st != AR_OK) return st;
        const uint64_t es = ar::esize_of(dtype);
        const uint64_t bytes = n * es;
        if (n == 0) return AR_OK;
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess) return AR_ERR_CUDA;
        bool aligned = true;
        st = ar::check_rank_buffers(P, n, static_cast<int>(es), dev, rank_bufs, true, &aligned);
        if (st != AR_OK) return st;
        if (P == 1) return AR_OK;

        ar::Lowered L;
        try {
            ar::lower(S, L);
        } catch (const std::length_error&) {
            return AR_ERR_UNSUPPORTED;
        }
        // the schedule's tables and partial slots must fit the static array
        std::vector<char> blob;
        const size_t o_progs = put(blob, L.progs), o_refs = put(blob, L.refs), o_ins = put(blob, L.ins);
        std::vector<size_t> o_sets;
        for (auto& s : L.sets) {
            o_sets.push_back(put(blob, s.bulk));
            o_sets.push_back(put(blob, s.edge));
            o_sets.push_back(put(blob, s.fallback));
        }
        if (blob.size() > kTableArea) return AR_ERR_UNSUPPORTED;
        uint64_t slot_stride = 0;
        if (S.params.form == AR_FORM_STEP && L.phys_slots > 1) {
            slot_stride = (bytes + 255) / 256 * 256;
            if (static_cast<uint64_t>(L.phys_slots - 1) * P * slot_stride > kSlotArea) return AR_ERR_UNSUPPORTED;
        }

        DeviceState* d = nullptr;
        st = setup(dev, d);
        if (st != AR_OK) return st;
        if (ar::prepare_kernels(dtype, op) != cudaSuccess) return AR_ERR_CUDA;
        const int smem_staged = ar::staged_smem_bytes(L);
        const int smem_stream = ar::stream_smem_bytes(L);
        const int smem_elem = (L.max_in_all + L.max_tmp_all) * ar::kElemThreads * 4;
        if (smem_staged > d->optin || smem_stream > d->optin || smem_elem > d->optin) return AR_ERR_UNSUPPORTED;

        cudaStream_t cs = static_cast<cudaStream_t>(stream);
        char* status = d->base;
        char* tables = d->base + kStatusArea;
        char* slots = tables + kTableArea;
        // the status word must start at zero; the tables are this call's
        if (cudaMemsetAsync(status, 0, sizeof(int), cs) != cudaSuccess) return AR_ERR_CUDA;
        if (cudaMemcpyAsync(tables, blob.data(), blob.size(), cudaMemcpyHostToDevice, cs) != cudaSuccess)
            return AR_ERR_CUDA;

        ar::KernelArgs a;
        std::memset(&a, 0, sizeof(a));
        for (int r = 0; r < P; ++r) a.bufs[r] = rank_bufs[r];
        a.scratch = slots;
        a.slot_stride = slot_stride;
        a.progs = reinterpret_cast<const ar::DevProg*>(tables + o_progs);
        a.refs = reinterpret_cast<const uint16_t*>(tables + o_refs);
        a.ins = reinterpret_cast<const uint32_t*>(tables + o_ins);
        a.status = reinterpret_cast<int*>(status);
        a.P = P;
        for (size_t i = 0; i < L.sets.size(); ++i) {
            const ar::LaunchSet& s = L.sets[i];
            const ar::WorkItem* bulk = reinterpret_cast<const ar::WorkItem*>(tables + o_sets[3 * i]);
            const ar::WorkItem* edge = reinterpret_cast<const ar::WorkItem*>(tables + o_sets[3 * i + 1]);
            const ar::WorkItem* fb = reinterpret_cast<const ar::WorkItem*>(tables + o_sets[3 * i + 2]);
            cudaError_t e = cudaSuccess;
            if (aligned && !s.small) {
                if (!s.bulk.empty()) {
                    a.items = bulk;
                    a.n_items = static_cast<uint32_t>(s.bulk.size());
                    const int grid = static_cast<int>(std::min<size_t>(s.bulk.size(), d->num_sms));
                    if (s.chain_words) {
                        const int cgrid =
                            static_cast<int>(std::min<size_t>(s.bulk.size(), ar::kChainWordCtasPerSm * d->num_sms));
                        e = ar::launch_chain_words(dtype, op, a, s.max_in, cgrid, cs);
                    } else if (s.copies) {
                        const int cgrid =
                            static_cast<int>(std::min<size_t>(s.bulk.size(), ar::kCopyCtasPerSm * d->num_sms));
                        e = ar::launch_copies(dtype, a, cgrid, cs);
                    } else if (s.few) {
                        const int cgrid =
                            static_cast<int>(std::min<size_t>(s.bulk.size(), ar::kCopyCtasPerSm * d->num_sms));
                        e = ar::launch_few(dtype, op, a, s.max_in, s.few_trees, cgrid, cs);
                    } else if (s.stream) {
                        a.tile_bytes = L.stream_tile;
                        a.stages = L.stream_stages;
                        a.flags = (s.tma_store ? ar::kArgTmaStore : 0) | (L.stream_trees ? ar::kArgTrees : 0) |
                                  (L.stream_tmem ? ar::kArgTmemStack : 0);
                        a.max_in = 1;
                        a.max_tmp = L.stream_slots;  // tree stack tiles after the stages
                        e = ar::launch_stream(dtype, op, a, grid, smem_stream, cs);
                    } else {
                        a.tile_bytes = L.tile_bytes;
                        a.stages = L.stages;
                        a.max_in = L.max_in;
                        a.max_tmp = L.max_tmp;
                        e = ar::launch_staged(dtype, op, a, grid, smem_staged, cs);
                    }
                }
                if (e == cudaSuccess && !s.edge.empty()) {
                    a.items = edge;
                    a.n_items = static_cast<uint32_t>(s.edge.size());
                    a.max_in = L.max_in_all;
                    a.max_tmp = L.max_tmp_all;
                    e = ar::launch_elementwise(dtype, op, a, smem_elem, cs);
                }
            } else if (!s.fallback.empty()) {
                a.items = fb;
                a.n_items = static_cast<uint32_t>(s.fallback.size());
                a.max_in = L.max_in_all;
                a.max_tmp = L.max_tmp_all;
                e = ar::launch_elementwise(dtype, op, a, smem_elem, cs);
            }
            if (e != cudaSuccess) return AR_ERR_CUDA;
        }
        return AR_OK;
    } catch (const std::bad_alloc&) {
        return AR_ERR_NOMEM;
    }
}

extern "C" ar_status ar_allreduce_static_check(void* stream) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return AR_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return AR_ERR_UNSUPPORTED;
    char* base = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_setup_mutex);
        if (g_dev[dev].ready) base = g_dev[dev].base;
    }
    if (!base) return AR_OK;  // no call has run on this device
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    int word = 0;
    cudaError_t e = cudaMemcpyAsync(&word, base, sizeof(int), cudaMemcpyDeviceToHost, cs);
    if (e == cudaSuccess) e = cudaStreamSynchronize(cs);
    if (e == cudaSuccess && word != 0) {
        e = cudaMemsetAsync(base, 0, sizeof(int), cs);
        if (e == cudaSuccess) e = cudaStreamSynchronize(cs);
    }
    if (e != cudaSuccess) return AR_ERR_CUDA;
    if (word & ar::kStatusBadProgram) return AR_ERR_INTERNAL;
    return word ? AR_ERR_TIMEOUT : AR_OK;
}
