// C ABI of the allreduce engine: argument checks, plan construction (compile,
// lower, upload) and launch dispatch.  No arithmetic of the allreduce happens
// here; every element is combined by the CUDA kernels.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstring>
#include <new>
#include <stdexcept>
#include <vector>

#include "ar.h"
#include "bufcheck.hpp"
#include "jit.hpp"
#include "kernels.hpp"
#include "lower.hpp"
#include "schedule.hpp"

namespace {
// AR_JIT_AUTO compiles a plan's DAG kernel when its staged launches move at
// least this much: smaller ones are launch-bound, where interpreting costs
// little and the compile time (a fraction of a second) would dominate.
constexpr uint64_t kJitMinBytes = 16ull << 20;
// Programs beyond this many instruction words stay interpreted: the
// compile time grows past a few seconds.
constexpr size_t kJitMaxWords = 4096;
// DAG programs with at least this many inputs run on the run-time compiled
// word kernel (registers) rather than the staged kernel (shared-memory
// tiles that shrink as the input count grows).
#ifndef AR_WORD_MIN_IN
#define AR_WORD_MIN_IN 33
#endif
constexpr int kWordMinIn = AR_WORD_MIN_IN;
// bf16 max / min programs, whose compare-and-selects make the evaluation
// ALU-heavy, go to the word kernel from this many inputs (its consumers read
// no staged tiles): measured at 64 MiB per rank, the word kernel 50-66% of
// the copy against 23-32% for the staged one at P = 28 ... 32, the staged
// one 72-77% against 53-57% at P = 20 / 24.
#ifndef AR_WORD_MIN_IN_SELECT
#define AR_WORD_MIN_IN_SELECT 25
#endif
// Guard bands around the step form's scratch: written with kGuardByte when
// the plan is created and compared by ar_plan_check, so a kernel that writes
// past either end of the scratch is reported rather than silently
// corrupting device memory.
constexpr size_t kGuardBytes = 256;
constexpr unsigned char kGuardByte = 0xA5;
}  // namespace

struct ar_schedule_s {
    ar::Schedule S;
};

struct ar_plan_s {
    ar::Schedule S;
    ar::Lowered L;
    int device = 0;
    int num_sms = 0;
    int smem_staged = 0;
    int smem_stream = 0;
    int smem_elem = 0;
    char* d_tables = nullptr;
    char* d_scratch_alloc = nullptr;  // [guard | scratch | guard]
    char* d_scratch = nullptr;
    uint64_t slot_stride = 0;
    uint64_t scratch_bytes = 0;
    int* d_status = nullptr;
    const void* dag_fn = nullptr;   // run-time compiled staged kernel, or null: interpret
    const void* word_fn = nullptr;  // run-time compiled word kernel (word sets need it)
    int word_grid = 0;              // its persistent grid: SMs x resident CTAs
    int smem_word = 0;              // its dynamic shared memory (prefetch stages)
    struct Set {
        const ar::WorkItem* bulk;
        const ar::WorkItem* edge;
        const ar::WorkItem* fallback;
        uint32_t n_bulk, n_edge, n_fallback;
        bool stream;
        bool small;
        bool tma_store;
        bool words;
        bool chain_words;
        bool copies;
        bool few;
        bool few_trees;
        bool chains;
        int max_in;
    };
    std::vector<Set> sets;
    // element windows of a fused plan for the pipelined host path
    using Window = ar::Window;
    std::vector<Window> windows;
    // copy streams of the pipelined host path, created on first use: the
    // copies of rank r go to stream r mod kCopyStreams in each direction
    static constexpr int kCopyStreams = 1;  // more streams measured slower on GB300
    cudaStream_t s_in[kCopyStreams] = {}, s_out[kCopyStreams] = {};
    std::vector<cudaEvent_t> events;  // (2 kCopyStreams + 1) per window + 1
    const ar::DevProg* d_progs = nullptr;
    const uint16_t* d_refs = nullptr;
    const uint32_t* d_ins = nullptr;
    // the last pointer set whose residency ar_execute checked and accepted
    std::vector<uintptr_t> checked;
};

namespace {

ar_status cuda_status(cudaError_t e) {
    if (e == cudaSuccess) return AR_OK;
    return e == cudaErrorMemoryAllocation ? AR_ERR_NOMEM : AR_ERR_CUDA;
}

void fill_info(const ar::Schedule& S, ar_plan_info* info) {
    std::memset(info, 0, sizeof(*info));
    const int es = ar::esize_of(S.dtype);
    info->P = S.P;
    info->dtype = S.dtype;
    info->op = S.op;
    info->algo = S.algo;
    info->form = S.params.form;
    info->order = S.params.order;
    info->phase = S.params.phase;
    info->n = static_cast<uint64_t>(S.n);
    info->steps = static_cast<int>(S.rounds.size());
    std::vector<uint64_t> per(S.P, 0);
    for (auto& rd : S.rounds)
        for (int r = 0; r < S.P; ++r) per[r] += static_cast<uint64_t>(rd.sent[r]) * es;
    for (uint64_t b : per) {
        info->sent_bytes_total += b;
        info->sent_bytes_max = std::max(info->sent_bytes_max, b);
    }
    info->combines = static_cast<uint64_t>(S.combines);
    for (auto& rd : S.rounds) info->messages += rd.xfers.size();
    info->max_slots = S.max_slots;
    info->n_segments = S.nseg();
}

template <class T>
size_t put(std::vector<char>& blob, const std::vector<T>& v) {
    size_t off = (blob.size() + 255) / 256 * 256;
    blob.resize(off + v.size() * sizeof(T));
    if (!v.empty()) std::memcpy(blob.data() + off, v.data(), v.size() * sizeof(T));
    return off;
}

void destroy_plan(ar_plan_s* p) {
    if (!p) return;
    for (cudaEvent_t e : p->events) cudaEventDestroy(e);
    for (int k = 0; k < ar_plan_s::kCopyStreams; ++k) {
        if (p->s_in[k]) cudaStreamDestroy(p->s_in[k]);
        if (p->s_out[k]) cudaStreamDestroy(p->s_out[k]);
    }
    if (p->d_tables) cudaFree(p->d_tables);
    if (p->d_scratch_alloc) cudaFree(p->d_scratch_alloc);
    if (p->d_status) cudaFree(p->d_status);
    delete p;
}

// The rank buffers of an execute: alignment and overlap every time; device
// residency and extent (ar::check_rank_buffers) whenever the pointer set
// differs from the last one accepted on this plan.
ar_status validate_bufs(ar_plan_s* plan, void* const* bufs, bool* aligned16) {
    const ar::Schedule& S = plan->S;
    const bool known = plan->checked.size() == static_cast<size_t>(S.P) &&
                       std::equal(plan->checked.begin(), plan->checked.end(), bufs,
                                  [](uintptr_t a, void* b) { return a == reinterpret_cast<uintptr_t>(b); });
    ar_status v = ar::check_rank_buffers(S.P, static_cast<uint64_t>(S.n), ar::esize_of(S.dtype), plan->device, bufs,
                                         !known, aligned16);
    if (v == AR_OK && !known) {
        plan->checked.clear();
        for (int r = 0; r < S.P; ++r) plan->checked.push_back(reinterpret_cast<uintptr_t>(bufs[r]));
    }
    return v;
}

void base_args(const ar_plan_s* plan, void* const* bufs, ar::KernelArgs& a) {
    std::memset(&a, 0, sizeof(a));
    for (int r = 0; r < plan->S.P; ++r) a.bufs[r] = bufs[r];
    a.scratch = plan->d_scratch;
    a.slot_stride = plan->slot_stride;
    a.progs = plan->d_progs;
    a.refs = plan->d_refs;
    a.ins = plan->d_ins;
    a.status = plan->d_status;
    a.P = plan->S.P;
}

// Launches bulk items [b0, b1) and edge items [e0, e1) of one set.
cudaError_t launch_range(const ar_plan_s* plan, ar::KernelArgs& a, const ar_plan_s::Set& s, uint32_t b0, uint32_t b1,
                         uint32_t e0, uint32_t e1, cudaStream_t st) {
    const ar::Schedule& S = plan->S;
    cudaError_t e = cudaSuccess;
    if (b1 > b0) {
        a.items = s.bulk + b0;
        a.n_items = b1 - b0;
        const int grid = static_cast<int>(std::min<uint32_t>(b1 - b0, plan->num_sms));
        if (s.words) {
            const int wgrid = static_cast<int>(std::min<uint32_t>(b1 - b0, plan->word_grid));
            e = ar::launch_dependent(plan->word_fn, wgrid, ar::kWordThreads, plan->smem_word, st, a);
        } else if (s.chain_words) {
            const int cgrid = static_cast<int>(std::min<uint32_t>(b1 - b0, plan->num_sms * ar::kChainWordCtasPerSm));
            e = ar::launch_chain_words(S.dtype, S.op, a, s.max_in, cgrid, st);
        } else if (s.copies) {
            const int cgrid = static_cast<int>(std::min<uint32_t>(b1 - b0, plan->num_sms * ar::kCopyCtasPerSm));
            e = ar::launch_copies(S.dtype, a, cgrid, st);
        } else if (s.few) {
            const int cgrid = static_cast<int>(std::min<uint32_t>(b1 - b0, plan->num_sms * ar::kCopyCtasPerSm));
            e = ar::launch_few(S.dtype, S.op, a, s.max_in, s.few_trees, cgrid, st);
        } else if (s.stream) {
            a.tile_bytes = plan->L.stream_tile;
            a.stages = plan->L.stream_stages;
            a.flags = (s.tma_store ? ar::kArgTmaStore : 0) | (plan->L.stream_trees ? ar::kArgTrees : 0) |
                      (plan->L.stream_tmem ? ar::kArgTmemStack : 0);
            a.max_in = 1;
            a.max_tmp = plan->L.stream_slots;  // tree stack tiles after the stages
            e = ar::launch_stream(S.dtype, S.op, a, grid, plan->smem_stream, st);
        } else {
            a.tile_bytes = plan->L.tile_bytes;
            a.stages = plan->L.stages;
            a.max_in = plan->L.max_in;
            a.max_tmp = plan->L.max_tmp;
            if (plan->dag_fn) {
                e = ar::launch_dependent(plan->dag_fn, grid, ar::kStagedThreads, plan->smem_staged, st, a);
            } else {
                e = ar::launch_staged(S.dtype, S.op, a, grid, plan->smem_staged, st);
            }
        }
    }
    if (e == cudaSuccess && e1 > e0) {
        a.items = s.edge + e0;
        a.n_items = e1 - e0;
        a.max_in = plan->L.max_in_all;
        a.max_tmp = plan->L.max_tmp_all;
        e = ar::launch_elementwise(S.dtype, S.op, a, plan->smem_elem, st);
    }
    return e;
}

// How a plan with this jit setting lowers: the word kernel for DAG sets when
// the run-time compiler is there (AUTO: for sets of at least kJitMinBytes).
// bf16 max / min programs from AR_WORD_MIN_IN_SELECT inputs on.
ar::LowerOptions lower_options(const ar::Schedule& S) {
    const int jit = S.params.jit;
    ar::LowerOptions lo;
    lo.jit_dag = jit != AR_JIT_OFF && ar::jit_available();
    lo.word_dag = lo.jit_dag;
    const bool selects = S.dtype == AR_BFLOAT16 && (S.op == AR_MAX || S.op == AR_MIN);
    lo.word_min_in = selects ? AR_WORD_MIN_IN_SELECT : kWordMinIn;
    lo.word_min_bytes = jit == AR_JIT_ON ? 0 : kJitMinBytes;
    return lo;
}

// Element windows for the pipelined host path (fused plans; ar::host_windows).
void make_windows(ar_plan_s* p) {
    p->windows.clear();
    if (p->L.sets.size() != 1) return;
    const uint64_t total = static_cast<uint64_t>(p->S.P) * p->S.n * ar::esize_of(p->S.dtype);
    p->windows = ar::host_windows(p->L.sets[0], p->S.n, total);
}

}  // namespace

extern "C" {

const char* ar_status_string(ar_status s) {
    switch (s) {
        case AR_OK: return "AR_OK: success";
        case AR_ERR_INVALID_ARG: return "AR_ERR_INVALID_ARG: invalid argument";
        case AR_ERR_UNSUPPORTED: return "AR_ERR_UNSUPPORTED: request not supported";
        case AR_ERR_CUDA: return "AR_ERR_CUDA: CUDA runtime error";
        case AR_ERR_NOMEM: return "AR_ERR_NOMEM: out of memory";
        case AR_ERR_TIMEOUT: return "AR_ERR_TIMEOUT: a bounded wait in a kernel gave up";
        case AR_ERR_INTERNAL: return "AR_ERR_INTERNAL: a kernel met a program it does not run, or wrote past the plan's scratch";
    }
    return "unknown ar_status";
}

ar_status ar_schedule_create(int P, uint64_t n, ar_dtype dtype, ar_op op, ar_algo algo, const ar_params* params,
                             ar_schedule_t* out) {
    if (!out) return AR_ERR_INVALID_ARG;
    *out = nullptr;
    if (n > (uint64_t(1) << 40)) return AR_ERR_UNSUPPORTED;
    try {
        auto* s = new ar_schedule_s();
        ar_status st = ar::compile_schedule(P, static_cast<int64_t>(n), dtype, op, algo, params, s->S);
        if (st != AR_OK) {
            delete s;
            return st;
        }
        *out = s;
        return AR_OK;
    } catch (const std::bad_alloc&) {
        return AR_ERR_NOMEM;
    }
}

ar_status ar_schedule_destroy(ar_schedule_t s) {
    delete s;
    return AR_OK;
}

ar_status ar_schedule_query(ar_schedule_t s, ar_plan_info* info) {
    if (!s || !info) return AR_ERR_INVALID_ARG;
    fill_info(s->S, info);
    return AR_OK;
}

ar_status ar_schedule_step_sent(ar_schedule_t s, int step, uint64_t* elems_per_rank) {
    if (!s || !elems_per_rank || step < 0 || step >= static_cast<int>(s->S.rounds.size()))
        return AR_ERR_INVALID_ARG;
    for (int r = 0; r < s->S.P; ++r) elems_per_rank[r] = static_cast<uint64_t>(s->S.rounds[step].sent[r]);
    return AR_OK;
}

ar_status ar_schedule_tree(ar_schedule_t s, int rank, uint64_t elem, char* buf, size_t cap, size_t* needed) {
    if (!s || rank < 0 || rank >= s->S.P || elem >= static_cast<uint64_t>(s->S.n)) return AR_ERR_INVALID_ARG;
    try {
        const int seg = s->S.seg_of(static_cast<int64_t>(elem));
        std::string t = s->S.dag.text(s->S.final_at(rank, seg));
        if (needed) *needed = t.size() + 1;
        if (!buf || cap < t.size() + 1) return AR_ERR_INVALID_ARG;
        std::memcpy(buf, t.c_str(), t.size() + 1);
        return AR_OK;
    } catch (const std::bad_alloc&) {
        return AR_ERR_NOMEM;
    }
}

ar_status ar_selftest_bounded_wait(uint32_t timeout_ms, void* stream) {
    if (timeout_ms < 1 || timeout_ms > 10000) return AR_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int* d_status = nullptr;
    cudaError_t e = cudaMalloc(&d_status, sizeof(int));
    if (e == cudaErrorMemoryAllocation) return AR_ERR_NOMEM;
    if (e == cudaSuccess) e = cudaMemsetAsync(d_status, 0, sizeof(int), st);
    if (e == cudaSuccess) e = ar::launch_wait_selftest(d_status, static_cast<uint64_t>(timeout_ms) * 1000000ull, st);
    int status = 0;
    if (e == cudaSuccess) e = cudaMemcpyAsync(&status, d_status, sizeof(int), cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    cudaFree(d_status);
    if (e != cudaSuccess) return cuda_status(e);
    return (status & ar::kStatusWaitFull) ? AR_ERR_TIMEOUT : AR_OK;
}

ar_status ar_schedule_dag_kernel(ar_schedule_t s, size_t* cubin_bytes) {
    if (!s || !cubin_bytes) return AR_ERR_INVALID_ARG;
    *cubin_bytes = 0;
    try {
        ar::Lowered L;
        ar::LowerOptions lo = lower_options(s->S);
        lo.jit_dag = lo.word_dag = true;  // both run-time kernels (a missing NVRTC is reported below)
        lo.word_min_bytes = 0;
        ar::lower(s->S, L, lo);
        for (const std::string& src : {ar::dag_kernel_source(s->S, L), ar::word_kernel_source(s->S, L)}) {
            if (src.empty()) continue;
            std::string cubin;
            const int rc = ar::compile_dag_kernel(src, cubin, nullptr);
            if (rc == 1) return AR_ERR_UNSUPPORTED;
            if (rc != 0) return AR_ERR_CUDA;
            *cubin_bytes += cubin.size();
        }
        return AR_OK;
    } catch (const std::length_error&) {
        return AR_ERR_UNSUPPORTED;
    } catch (const std::bad_alloc&) {
        return AR_ERR_NOMEM;
    }
}

ar_status ar_schedule_lowering(ar_schedule_t s, ar_lowering_info* out) {
    if (!s || !out) return AR_ERR_INVALID_ARG;
    *out = ar_lowering_info{};
    try {
        ar::Lowered L;
        ar::lower(s->S, L, lower_options(s->S));
        const int es = ar::esize_of(s->S.dtype);
        std::vector<ar::Window> W;
        if (L.sets.size() == 1)
            W = ar::host_windows(L.sets[0], s->S.n, static_cast<uint64_t>(s->S.P) * s->S.n * es);
        const ar::LoweringCheck c = ar::check_lowering(L, s->S.n, es, W);
        out->items = c.items;
        out->launch_sets = static_cast<int>(L.sets.size());
        out->windows = static_cast<int>(W.size());
        out->tiling_ok = c.tiling_ok;
        out->windows_ok = c.windows_ok;
        out->wave_balance = c.wave_balance;
        out->stream_tile_bytes = L.stream_tile;
        out->stream_stages = L.stream_stages;
        out->staged_tile_bytes = L.tile_bytes;
        out->staged_stages = L.stages;
        out->dag_words = ar::dag_kernel_words(L);
        out->word_kernel_words = ar::word_kernel_words(L);
        out->stream_tmem = L.stream_tmem ? 1 : 0;
        for (const ar::LaunchSet& ls : L.sets) {
            out->word_sets += ls.words;
            out->copy_sets += ls.copies;
            out->few_sets += ls.few;
        }
        return AR_OK;
    } catch (const std::bad_alloc&) {
        return AR_ERR_NOMEM;
    }
}

ar_status ar_plan_create(int P, uint64_t n, ar_dtype dtype, ar_op op, ar_algo algo, const ar_params* params,
                         ar_plan_t* out) {
    ar::TraceRange trace("ar_plan_create");
    if (!out) return AR_ERR_INVALID_ARG;
    *out = nullptr;
    if (n > (uint64_t(1) << 40)) return AR_ERR_UNSUPPORTED;
    ar_plan_s* p = nullptr;
    try {
        p = new ar_plan_s();
        ar_status st = ar::compile_schedule(P, static_cast<int64_t>(n), dtype, op, algo, params, p->S);
        if (st != AR_OK) {
            delete p;
            return st;
        }
        ar::LowerOptions lo = lower_options(p->S);
        try {
            ar::lower(p->S, p->L, lo);
        } catch (const std::length_error&) {
            delete p;
            return AR_ERR_UNSUPPORTED;
        }
        cudaError_t e = cudaGetDevice(&p->device);
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&p->num_sms, cudaDevAttrMultiProcessorCount, p->device);
        int optin = 0;
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, p->device);
        if (e == cudaSuccess) e = ar::prepare_kernels(dtype, op);
        if (e != cudaSuccess) {
            delete p;
            return cuda_status(e);
        }
        // the word-kernel sets' programs as run-time compiled code; without
        // it (no NVRTC, too many instruction words, a failed compile) the
        // plan is lowered again with those sets on the staged kernel
        const size_t wwords = ar::word_kernel_words(p->L);
        if (wwords > 0) {
            p->smem_word = ar::word_kernel_prefetch(p->L) ? ar::word_kernel_smem(ar::word_kernel_max_in(p->L)) : 0;
            if (wwords <= kJitMaxWords && p->smem_word <= optin)
                p->word_fn = ar::load_dag_kernel(ar::word_kernel_source(p->S, p->L), "ar_word_kernel");
            int nb = 0;
            if (p->word_fn &&
                cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, p->word_fn, ar::kWordThreads, p->smem_word) ==
                    cudaSuccess &&
                nb > 0) {
                p->word_grid = p->num_sms * nb;
            } else {
                cudaGetLastError();
                p->word_fn = nullptr;
                lo.word_dag = false;
                ar::lower(p->S, p->L, lo);
            }
        }
        const ar::Lowered& L = p->L;
        p->smem_staged = ar::staged_smem_bytes(L);
        p->smem_stream = ar::stream_smem_bytes(L);
        p->smem_elem = (L.max_in_all + L.max_tmp_all) * ar::kElemThreads * 4;
        if (p->smem_staged > optin || p->smem_stream > optin || p->smem_elem > optin) {
            delete p;
            return AR_ERR_UNSUPPORTED;
        }
        // the staged launches' DAG programs as run-time compiled code; a plan
        // lowered for compiled programs (no shared-memory temporaries) that
        // is not compiled after all is lowered again for the interpreter
        const size_t words = ar::dag_kernel_words(L);
        if (words > 0 && words <= kJitMaxWords && p->S.params.jit != AR_JIT_OFF) {
            uint64_t dag_bytes = 0;
            for (const ar::LaunchSet& s : L.sets)
                if (!s.stream && !s.small && !s.words && !s.chain_words && !s.copies && !s.few && !s.bulk.empty())
                    dag_bytes += s.bytes;
            if (p->S.params.jit == AR_JIT_ON || dag_bytes >= kJitMinBytes)
                p->dag_fn = ar::load_dag_kernel(ar::dag_kernel_source(p->S, L));
        }
        if (!p->dag_fn && lo.jit_dag && words > 0) {
            lo.jit_dag = false;
            ar::lower(p->S, p->L, lo);
            p->smem_staged = ar::staged_smem_bytes(L);
            p->smem_elem = (L.max_in_all + L.max_tmp_all) * ar::kElemThreads * 4;
            if (p->smem_staged > optin || p->smem_elem > optin) {
                delete p;
                return AR_ERR_UNSUPPORTED;
            }
        }
        // one device blob: programs, refs, instructions, then every item list
        std::vector<char> blob;
        size_t o_progs = put(blob, L.progs), o_refs = put(blob, L.refs), o_ins = put(blob, L.ins);
        std::vector<size_t> o_sets;
        for (auto& s : L.sets) {
            o_sets.push_back(put(blob, s.bulk));
            o_sets.push_back(put(blob, s.edge));
            o_sets.push_back(put(blob, s.fallback));
        }
        blob.resize(std::max<size_t>(blob.size(), 256));
        e = cudaMalloc(&p->d_tables, blob.size());
        if (e == cudaSuccess) e = cudaMemcpy(p->d_tables, blob.data(), blob.size(), cudaMemcpyHostToDevice);
        if (e == cudaSuccess) e = cudaMalloc(&p->d_status, 256);
        if (e == cudaSuccess) e = cudaMemset(p->d_status, 0, 256);
        const int es = ar::esize_of(dtype);
        if (e == cudaSuccess && p->S.params.form == AR_FORM_STEP && L.phys_slots > 1) {
            // second partials and the twins of versioned rounds, per rank
            p->slot_stride = (static_cast<uint64_t>(n) * es + 255) / 256 * 256;
            p->scratch_bytes = static_cast<uint64_t>(L.phys_slots - 1) * P * p->slot_stride;
            e = cudaMalloc(&p->d_scratch_alloc, p->scratch_bytes + 2 * kGuardBytes);
            if (e == cudaSuccess) {
                p->d_scratch = p->d_scratch_alloc + kGuardBytes;
                e = cudaMemset(p->d_scratch_alloc, kGuardByte, kGuardBytes);
            }
            if (e == cudaSuccess) e = cudaMemset(p->d_scratch + p->scratch_bytes, kGuardByte, kGuardBytes);
        }
        if (e != cudaSuccess) {
            destroy_plan(p);
            return cuda_status(e);
        }
        p->d_progs = reinterpret_cast<const ar::DevProg*>(p->d_tables + o_progs);
        p->d_refs = reinterpret_cast<const uint16_t*>(p->d_tables + o_refs);
        p->d_ins = reinterpret_cast<const uint32_t*>(p->d_tables + o_ins);
        for (size_t i = 0; i < L.sets.size(); ++i) {
            ar_plan_s::Set s;
            s.bulk = reinterpret_cast<const ar::WorkItem*>(p->d_tables + o_sets[3 * i]);
            s.edge = reinterpret_cast<const ar::WorkItem*>(p->d_tables + o_sets[3 * i + 1]);
            s.fallback = reinterpret_cast<const ar::WorkItem*>(p->d_tables + o_sets[3 * i + 2]);
            s.n_bulk = static_cast<uint32_t>(L.sets[i].bulk.size());
            s.n_edge = static_cast<uint32_t>(L.sets[i].edge.size());
            s.n_fallback = static_cast<uint32_t>(L.sets[i].fallback.size());
            s.stream = L.sets[i].stream;
            s.small = L.sets[i].small;
            s.tma_store = L.sets[i].tma_store;
            s.words = L.sets[i].words;
            s.chain_words = L.sets[i].chain_words;
            s.copies = L.sets[i].copies;
            s.few = L.sets[i].few;
            s.few_trees = L.sets[i].few_trees;
            s.max_in = L.sets[i].max_in;
            s.chains = L.sets[i].chains;
            p->sets.push_back(s);
        }
        make_windows(p);
        *out = p;
        return AR_OK;
    } catch (const std::bad_alloc&) {
        destroy_plan(p);
        return AR_ERR_NOMEM;
    }
}

ar_status ar_plan_destroy(ar_plan_t plan) {
    if (!plan) return AR_ERR_INVALID_ARG;
    cudaError_t e = cudaDeviceSynchronize();
    destroy_plan(plan);
    return cuda_status(e);
}

ar_status ar_plan_query(ar_plan_t plan, ar_plan_info* info) {
    if (!plan || !info) return AR_ERR_INVALID_ARG;
    fill_info(plan->S, info);
    info->hbm_bytes = plan->L.hbm_bytes;
    info->scratch_bytes = plan->scratch_bytes;
    info->launches = plan->L.launches;
    info->tile_bytes = plan->L.tile_bytes;
    info->n_programs = static_cast<int>(plan->L.progs.size());
    info->n_items = plan->L.n_items;
    for (const ar::LaunchSet& s : plan->L.sets) {
        if (s.small) {
            info->kernels |= AR_KERNEL_ELEMENTWISE;
            continue;
        }
        if (!s.bulk.empty())
            info->kernels |= s.words         ? AR_KERNEL_WORD_JIT
                             : s.chain_words ? AR_KERNEL_CHAIN_WORD
                             : s.copies      ? AR_KERNEL_COPY
                             : s.few         ? AR_KERNEL_FEW
                             : s.stream      ? AR_KERNEL_STREAM
                                             : AR_KERNEL_STAGED;
        if (!s.bulk.empty() && !s.stream && !s.words && !s.chain_words && !s.copies && !s.few && plan->dag_fn)
            info->kernels |= AR_KERNEL_DAG_JIT;
        if (!s.edge.empty()) info->kernels |= AR_KERNEL_ELEMENTWISE;
    }
    return AR_OK;
}

ar_status ar_plan_check_buffers(ar_plan_t plan, void* const* rank_bufs) {
    if (!plan || !rank_bufs) return AR_ERR_INVALID_ARG;
    const ar::Schedule& S = plan->S;
    if (S.n == 0) return AR_OK;
    bool aligned = false;
    return ar::check_rank_buffers(S.P, static_cast<uint64_t>(S.n), ar::esize_of(S.dtype), plan->device, rank_bufs,
                                  true, &aligned);
}

ar_status ar_execute(ar_plan_t plan, void* const* rank_bufs, void* stream) {
    ar::TraceRange trace("ar_execute");
    if (!plan || !rank_bufs) return AR_ERR_INVALID_ARG;
    const ar::Schedule& S = plan->S;
    if (S.n == 0) return AR_OK;  // nothing to touch: any pointers are accepted
    bool aligned = false;
    ar_status v = validate_bufs(plan, rank_bufs, &aligned);
    if (v != AR_OK) return v;
    if (S.P == 1) return AR_OK;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    ar::KernelArgs a;
    base_args(plan, rank_bufs, a);
    // buffers off 16-byte alignment: chains of 4-byte elements (every
    // element on a 32-bit word) on the chain word kernel, the rest element
    // by element
    const bool words_ok = ar::esize_of(S.dtype) == 4;
    for (const auto& s : plan->sets) {
        cudaError_t e = cudaSuccess;
        if (aligned && !s.small) {
            e = launch_range(plan, a, s, 0, s.n_bulk, 0, s.n_edge, st);
        } else if (s.n_fallback && !aligned && !s.small && words_ok && s.chains) {
            a.items = s.fallback;
            a.n_items = s.n_fallback;
            const int cgrid = static_cast<int>(std::min<uint32_t>(s.n_fallback, plan->num_sms * ar::kChainWordCtasPerSm));
            e = ar::launch_chain_words(S.dtype, S.op, a, s.max_in, cgrid, st);
        } else if (s.n_fallback) {
            a.items = s.fallback;
            a.n_items = s.n_fallback;
            a.max_in = plan->L.max_in_all;
            a.max_tmp = plan->L.max_tmp_all;
            e = ar::launch_elementwise(S.dtype, S.op, a, plan->smem_elem, st);
        }
        if (e != cudaSuccess) return cuda_status(e);
    }
    return AR_OK;
}

ar_status ar_execute_host(ar_plan_t plan, void* const* host_bufs, void* const* dev_bufs, void* stream) {
    ar::TraceRange trace("ar_execute_host");
    if (!plan || !host_bufs || !dev_bufs) return AR_ERR_INVALID_ARG;
    const ar::Schedule& S = plan->S;
    const int P = S.P;
    const size_t es = ar::esize_of(S.dtype);
    const size_t bytes = static_cast<size_t>(S.n) * es;
    for (int r = 0; r < P; ++r)
        if (!host_bufs[r]) return AR_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    bool aligned = false;
    if (S.n > 0) {
        ar_status v = validate_bufs(plan, dev_bufs, &aligned);
        if (v != AR_OK) return v;
    }
    if (!aligned || plan->windows.size() < 2 || P == 1) {
        // one pass: every copy in, the allreduce, every copy out
        for (int r = 0; r < P; ++r) {
            cudaError_t e = cudaMemcpyAsync(dev_bufs[r], host_bufs[r], bytes, cudaMemcpyHostToDevice, st);
            if (e != cudaSuccess) return cuda_status(e);
        }
        ar_status s = ar_execute(plan, dev_bufs, stream);
        if (s != AR_OK) return s;
        for (int r = 0; r < P; ++r) {
            cudaError_t e = cudaMemcpyAsync(host_bufs[r], dev_bufs[r], bytes, cudaMemcpyDeviceToHost, st);
            if (e != cudaSuccess) return cuda_status(e);
        }
        return cuda_status(cudaStreamSynchronize(st));
    }
    // Pipelined: every element's reduction depends only on that element of
    // every rank, so the buffers are processed in windows.  Window w's copies
    // in run on the s_in streams, its reduction on `stream`, its copies out on
    // the s_out streams; copies of neighbouring windows overlap the reduction
    // of window w, and the per-rank copies of a window spread over several
    // streams (copy engines) in each direction.
    constexpr int K = ar_plan_s::kCopyStreams;
    const size_t W = plan->windows.size();
    const size_t per_win = 2 * K + 1;
    cudaError_t e = cudaSuccess;
    if (plan->events.size() != per_win * W + 1) {
        for (int k = 0; k < K && e == cudaSuccess; ++k) {
            if (!plan->s_in[k]) e = cudaStreamCreateWithFlags(&plan->s_in[k], cudaStreamNonBlocking);
            if (e == cudaSuccess && !plan->s_out[k]) e = cudaStreamCreateWithFlags(&plan->s_out[k], cudaStreamNonBlocking);
        }
        for (cudaEvent_t x : plan->events) cudaEventDestroy(x);
        plan->events.clear();
        for (size_t k = 0; e == cudaSuccess && k < per_win * W + 1; ++k) {
            cudaEvent_t ev;
            e = cudaEventCreateWithFlags(&ev, cudaEventDisableTiming);
            if (e == cudaSuccess) plan->events.push_back(ev);
        }
        if (e != cudaSuccess) return cuda_status(e);
    }
    cudaEvent_t* ev = plan->events.data();
    cudaEvent_t start = ev[per_win * W];
    auto chk = [&](cudaError_t x) {
        if (e == cudaSuccess) e = x;
    };
    chk(cudaEventRecord(start, st));
    for (int k = 0; k < K; ++k) {
        chk(cudaStreamWaitEvent(plan->s_in[k], start, 0));
        chk(cudaStreamWaitEvent(plan->s_out[k], start, 0));
    }
    ar::KernelArgs a;
    base_args(plan, dev_bufs, a);
    const ar_plan_s::Set& set = plan->sets[0];
    for (size_t w = 0; w < W && e == cudaSuccess; ++w) {
        const ar_plan_s::Window& win = plan->windows[w];
        cudaEvent_t* in_done = ev + per_win * w;      // K events
        cudaEvent_t reduced = ev[per_win * w + K];
        cudaEvent_t* out_done = ev + per_win * w + K + 1;  // K events
        if (win.lo < 0 || win.hi <= win.lo || win.hi > S.n) {  // never a copy outside the buffers
            e = cudaErrorInvalidValue;
            break;
        }
        const size_t off = static_cast<size_t>(win.lo) * es, len = static_cast<size_t>(win.hi - win.lo) * es;
        for (int r = 0; r < P; ++r)
            chk(cudaMemcpyAsync(static_cast<char*>(dev_bufs[r]) + off, static_cast<const char*>(host_bufs[r]) + off,
                                len, cudaMemcpyHostToDevice, plan->s_in[r % K]));
        for (int k = 0; k < K; ++k) {
            chk(cudaEventRecord(in_done[k], plan->s_in[k]));
            chk(cudaStreamWaitEvent(st, in_done[k], 0));
        }
        if (e == cudaSuccess) e = launch_range(plan, a, set, win.b0, win.b1, win.e0, win.e1, st);
        chk(cudaEventRecord(reduced, st));
        for (int k = 0; k < K; ++k) chk(cudaStreamWaitEvent(plan->s_out[k], reduced, 0));
        for (int r = 0; r < P; ++r)
            chk(cudaMemcpyAsync(static_cast<char*>(host_bufs[r]) + off, static_cast<const char*>(dev_bufs[r]) + off,
                                len, cudaMemcpyDeviceToHost, plan->s_out[r % K]));
        for (int k = 0; k < K; ++k) chk(cudaEventRecord(out_done[k], plan->s_out[k]));
    }
    if (e == cudaSuccess)
        for (int k = 0; k < K; ++k) chk(cudaStreamWaitEvent(st, ev[per_win * (W - 1) + K + 1 + k], 0));
    chk(cudaStreamSynchronize(st));
    return cuda_status(e);
}

ar_status ar_plan_check(ar_plan_t plan) {
    if (!plan) return AR_ERR_INVALID_ARG;
    cudaError_t e = cudaDeviceSynchronize();
    int word = 0;
    if (e == cudaSuccess) e = cudaMemcpy(&word, plan->d_status, sizeof(int), cudaMemcpyDeviceToHost);
    bool guards_ok = true;
    if (e == cudaSuccess && plan->d_scratch_alloc) {
        unsigned char g[2 * kGuardBytes];
        e = cudaMemcpy(g, plan->d_scratch_alloc, kGuardBytes, cudaMemcpyDeviceToHost);
        if (e == cudaSuccess)
            e = cudaMemcpy(g + kGuardBytes, plan->d_scratch + plan->scratch_bytes, kGuardBytes, cudaMemcpyDeviceToHost);
        for (size_t i = 0; e == cudaSuccess && i < sizeof(g); ++i) guards_ok = guards_ok && g[i] == kGuardByte;
    }
    if (e != cudaSuccess) return cuda_status(e);
    if (word != 0) cudaMemset(plan->d_status, 0, sizeof(int));
    if (!guards_ok || (word & ar::kStatusBadProgram)) return AR_ERR_INTERNAL;
    if (word != 0) return AR_ERR_TIMEOUT;
    return AR_OK;
}

}  // extern "C"
