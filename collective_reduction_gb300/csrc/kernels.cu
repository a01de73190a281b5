// CUDA kernels of the allreduce engine (sm_103a).
//
// stream_kernel: the hot path (chains, single trees and fp32 accumulation:
// the fused pass of every schedule whose ranks share one tree per element,
// and the step form's rounds of independent transfers).  Persistent, one CTA
// per SM, warp-specialised: warp 0 resolves source addresses and its lane 0
// issues one cp.async.bulk (TMA bulk copy, L2 evict-first) per rank tile into
// a ring of shared-memory stages, each completing on its own mbarrier; eight
// consumer warps fold every rank tile into per-thread register accumulators
// in program order (a tree keeps its deeper stack entries in shared-memory
// tiles after the stages) and, after the item's last input, store the result
// to every output with 128-bit streaming stores or TMA bulk stores.  Rank
// tiles are 32 KB (16 KB for bf16 fp32 accumulation and deep trees) whatever
// P is, so all consumer threads stay busy and ~200 KB per SM is in flight.
//
// staged_kernel: for DAG programs (rank-specific results) and for chains
// whose rank tiles would be tiny.  Same structure, but a stage holds all
// input tiles of one item, which the consumers evaluate as straight-line
// instructions with shared-memory temporaries (the plan's DAG programs can
// instead run as compiled code: the same loop, compiled per plan at run time
// from device.cuh).
//
// Every wait is bounded: after two seconds the waiter sets a bit in the
// status word and the CTA winds down (a failing producer first waits, again
// bounded, for its copies in flight).
//
// elementwise_kernel: one CTA per work item, one element per thread (the
// CTA's threads load the item's inputs together); used for small passes, the
// unaligned heads / tails of ranges and buffers that are not 16-byte
// aligned.  Same programs, same arithmetic, same accumulation order.
//
// Element arithmetic (sum / prod / max / min over int32, fp32, bf16): int32
// wraps, fp32 uses IEEE round-to-nearest-even adds and multiplies without
// contraction or flushing, bf16 widens to fp32, applies the fp32 op and
// rounds back to bf16 to nearest even after every op; max is a > b ? a : b
// and min a < b ? a : b.
#include <cstdint>

#include "device.cuh"
#include "kernels.hpp"

namespace ar {
namespace {

template <int DT, int OP>
__global__ void __launch_bounds__(kStagedThreads, 1) staged_kernel(const __grid_constant__ KernelArgs a) {
    extern __shared__ __align__(128) uint8_t smem[];
    staged_body<DT, OP>(a, smem, [&](const Stage& sm, const DevProg& pg, uint32_t, uint32_t st, uint32_t nvec,
                                     int64_t off, int ct) { dag_item<DT, OP>(a, pg, st, sm.tmps, nvec, off, ct); });
}

// ---------------------------------------------------- rank-streaming kernel
//
// For programs that are a chain, a single tree or an fp32 accumulation (the
// ring's fused pass and rounds, the fused trees of the other schedules,
// every FP32ACC pass) the inputs are consumed strictly in order, so an
// item's tiles need not be resident together: the producer streams one rank
// tile (VPT vectors per consumer thread) per stage through a ring of stages
// (as many as the lowering asks for), and each consumer thread keeps its
// vectors' accumulators in registers across the item's inputs.  Tile size
// and thread utilisation do not shrink with P.

template <int ES>
__device__ void stream_produce(const KernelArgs& a, const Stage& sm) {
    const uint32_t lane = threadIdx.x & 31u;
    const uint64_t policy = AR_L2_EVICT_FIRST ? evict_first_policy() : 0;
    uint32_t g = 0;  // rank tiles issued so far
    bool ok = true;
    for (uint32_t it = blockIdx.x; it < a.n_items && ok; it += gridDim.x) {
        const WorkItem w = a.items[it];
        const DevProg pg = a.progs[w.prog];
        const uint32_t nb = w.count * ES;
        const int64_t off = w.elem * ES;
        for (uint32_t i0 = 0; i0 < pg.n_in && ok; i0 += 32) {
            // the warp resolves 32 source addresses at once; lane 0 issues
            const char* mine = nullptr;
            if (i0 + lane < pg.n_in) mine = buf_addr(a, a.refs[pg.in_off + i0 + lane]) + off;
            const uint32_t cnt = min(32u, pg.n_in - i0);
            for (uint32_t j = 0; j < cnt; ++j) {
                const char* src = reinterpret_cast<const char*>(
                    __shfl_sync(0xFFFFFFFFu, reinterpret_cast<unsigned long long>(mine), j));
                int issued = 0;
                if (lane == 0) {
                    const uint32_t s = g % a.stages, ph = (g / a.stages) & 1u;
                    if (mbar_wait(sm.empty + 8 * s, ph ^ 1u)) {
                        const uint32_t bar = sm.full + 8 * s;
                        mbar_expect_tx(bar, nb);
                        bulk_load(sm.tiles + s * a.tile_bytes, src, nb, bar, policy);
                        issued = 1;
                    }
                }
                issued = __shfl_sync(0xFFFFFFFFu, issued, 0);
                if (!issued) {
                    ok = false;
                    break;
                }
                ++g;
            }
        }
    }
    if (!ok && lane == 0) {
        atomicOr(a.status, kStatusWaitEmpty);
        const uint32_t first = g > static_cast<uint32_t>(a.stages) ? g - a.stages : 0;
        for (uint32_t j = first; j < g; ++j)
            if (!mbar_wait(sm.full + 8 * (j % a.stages), (j / a.stages) & 1u)) atomicOr(a.status, kStatusDrain);
    }
}

// warp 0 produces, warp 1 stores (TMA-store epilogue only), the rest consume
constexpr int kStreamLead = 2;
constexpr int kStreamThreads = 32 * (kStreamLead + kConsumerWarps);
// tensor-memory tree stack: all 512 columns (two consumer warps per lane
// quarter, 256 columns = 8 entries of 32 each), the allocated address kept in
// the last word of the barrier area (full / ready / empty barriers take 24
// bytes per stage, at most kMaxStreamStages stages)
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemAddrOffset = kBarrierBytes - 8;
static_assert(kTmemAddrOffset >= 24 * (kBarrierBytes / 24), "the barrier area's last word is free");

__device__ __forceinline__ void mbar_arrive_count(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// global <- shared bulk copy (TMA store), tracked by the issuing thread's
// bulk async-groups
__device__ __forceinline__ void bulk_store(char* dst, uint32_t src, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(src), "r"(bytes)
                 : "memory");
}

// Storer (lane 0 of warp 1): once the consumers have written an item's
// result into the stage of its last rank tile, copy that tile to every
// output buffer, and release the stage when the copies have read it.
//
// There is one `ready` barrier per stage: a stage holding an item's last tile
// is refilled only after the storer has released it, so no consumer warp can
// arrive twice within one phase of that stage's barrier.  ready_parity keeps
// the phase parity of every stage's barrier.
template <int ES>
__device__ void stream_store(const KernelArgs& a, const Stage& sm) {
    uint32_t g = 0, ready_parity = 0;
    for (uint32_t it = blockIdx.x; it < a.n_items; it += gridDim.x) {
        const WorkItem w = a.items[it];
        const DevProg pg = a.progs[w.prog];
        g += pg.n_in;
        const uint32_t s = (g - 1) % a.stages;
        if (!mbar_wait(sm.ready + 8 * s, (ready_parity >> s) & 1u)) {
            atomicOr(a.status, kStatusWaitFull);
            break;
        }
        ready_parity ^= 1u << s;
        const uint32_t src = sm.tiles + s * a.tile_bytes;
        const uint32_t nb = w.count * ES;
        const int64_t off = w.elem * ES;
        for (uint32_t o = 0; o < pg.n_out; ++o) bulk_store(out_addr(a, pg, o) + off, src, nb);
        asm volatile("cp.async.bulk.commit_group;" ::: "memory");
        asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
        mbar_arrive_count(sm.empty + 8 * s, kConsumerWarps);
    }
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// Waits for rank tile g; its shared address, or 0 after the bounded wait.
__device__ __forceinline__ uint32_t stream_acquire(const KernelArgs& a, const Stage& sm, uint32_t g) {
    const uint32_t s = g % a.stages, ph = (g / a.stages) & 1u;
    if (!mbar_wait(sm.full + 8 * s, ph)) {
        atomicOr(a.status, kStatusWaitFull);
        return 0;
    }
    return sm.tiles + s * a.tile_bytes;
}

// After a tile that is not an item's last input: give the stage back.
__device__ __forceinline__ void stream_release(const KernelArgs& a, const Stage& sm, uint32_t g, int lane) {
    __syncwarp();
    if (lane == 0) mbar_arrive(sm.empty + 8 * (g % a.stages));
}

// After an item's last input: with TMA stores, write the result over this
// thread's own vectors of the tile and hand the stage to the storer (which
// copies it to every output and then gives the stage back); otherwise give
// the stage back and store the result directly.
template <int VPT>
__device__ __forceinline__ void stream_finish(const KernelArgs& a, const Stage& sm, uint32_t g, uint32_t t,
                                              const DevProg& pg, int64_t off, uint32_t nvec, int ct,
                                              const uint4 (&res)[VPT]) {
    const int lane = ct & 31;
    if (a.flags & kArgTmaStore) {
#pragma unroll
        for (int j = 0; j < VPT; ++j) {
            const uint32_t v = ct + j * kConsumers;
            if (v < nvec) sts128(t + v * 16, res[j]);
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        if (lane == 0) mbar_arrive(sm.ready + 8 * (g % a.stages));
    } else {
        stream_release(a, sm, g, lane);
        for (uint32_t o = 0; o < pg.n_out; ++o) {
            char* dst = out_addr(a, pg, o) + off;
#pragma unroll
            for (int j = 0; j < VPT; ++j) {
                const uint32_t v = ct + j * kConsumers;
                if (v < nvec) stg128(dst + v * 16, res[j]);
            }
        }
    }
}

// A single tree streamed one leaf tile at a time.  The top of the stack
// stays in registers (acc); the entries below it live in the shared-memory
// stack tiles (entry k in tile k, this thread's own vectors only, so no
// barrier is needed).  After a leaf arrives: with no combine to follow, the
// old top moves to shared memory and the leaf becomes the top; otherwise the
// first combine takes the leaf straight from its stage (top (+) leaf) and
// the rest fold shared-memory entries into the top (entry (+) top: the left
// operand is the deeper one).  FULL: the item covers a whole tile, so every
// thread's VPT vectors are in range and the bounds test is left out.
//
// TM: the stack entries below the top live in tensor memory instead (tstack:
// this warp's lanes and columns; 32 columns per entry, one tcgen05.st / ld per
// push / pop, by the whole warp, every vector alike).
template <int DT, int OP, int VPT, bool FULL, bool TM>
__device__ __forceinline__ bool stream_tree(const KernelArgs& a, const Stage& sm, const DevProg& pg, uint32_t& g,
                                            int64_t off, uint32_t nvec, int ct, uint32_t tstack) {
    static_assert(!TM || VPT == 8, "the TMEM stack moves 8 vectors per entry");
    const int lane = ct & 31;
    if (pg.n_tmp > static_cast<uint32_t>(a.max_tmp)) {  // deeper than the launch's stack
        atomicOr(a.status, kStatusBadProgram);
        return false;
    }
    uint4 acc[VPT];
    uint32_t sp = 0;  // stack entries, the top one in acc
    for (uint32_t i = 0; i < pg.n_in; ++i, ++g) {
        const uint32_t t = stream_acquire(a, sm, g);
        if (!t) return false;
        uint32_t c = (a.ins[pg.ins_off + (i >> 3)] >> (4 * (i & 7))) & 15u;
        if (sp == 0 || c == 0) {
            if (sp > 0) {
                if constexpr (TM) {
                    tmem_store32(tstack + (sp - 1) * 32u, acc);
                } else {
                    const uint32_t slot = sm.tmps + (sp - 1) * a.tile_bytes;
#pragma unroll
                    for (int j = 0; j < VPT; ++j) {
                        const uint32_t v = ct + j * kConsumers;
                        if (FULL || v < nvec) sts128(slot + v * 16, acc[j]);
                    }
                }
            }
#pragma unroll
            for (int j = 0; j < VPT; ++j) {
                const uint32_t v = ct + j * kConsumers;
                if (FULL || v < nvec) acc[j] = lds128(t + v * 16);
            }
            ++sp;
        } else {
#pragma unroll
            for (int j = 0; j < VPT; ++j) {
                const uint32_t v = ct + j * kConsumers;
                if (FULL || v < nvec) acc[j] = vop<DT, OP>(acc[j], lds128(t + v * 16));
            }
            --c;
        }
        for (; c > 0; --c, --sp) {
            if constexpr (TM) {
                uint4 e[VPT];
                tmem_load32(tstack + (sp - 2) * 32u, e);
#pragma unroll
                for (int j = 0; j < VPT; ++j) acc[j] = vop<DT, OP>(e[j], acc[j]);
            } else {
                const uint32_t slot = sm.tmps + (sp - 2) * a.tile_bytes;
#pragma unroll
                for (int j = 0; j < VPT; ++j) {
                    const uint32_t v = ct + j * kConsumers;
                    if (FULL || v < nvec) acc[j] = vop<DT, OP>(lds128(slot + v * 16), acc[j]);
                }
            }
        }
        if (i + 1 < pg.n_in) {
            stream_release(a, sm, g, lane);
        } else {
            if (pg.flags & PF_AVG) {
#pragma unroll
                for (int j = 0; j < VPT; ++j) acc[j] = vdiv<DT>(acc[j], static_cast<float>(a.P));
            }
            stream_finish<VPT>(a, sm, g, t, pg, off, nvec, ct, acc);
        }
    }
    return true;
}

// TREES: the instantiation for launches with single-tree programs (chains
// and trees); the others run chains and fp32 accumulation.  Keeping the tree
// stack and the accumulators in separate instantiations keeps each within
// the register budget.
template <int DT, int OP, int VPT, bool TREES, bool TM>
__device__ void stream_consume(const KernelArgs& a, const Stage& sm, int ct, uint32_t tstack) {
    constexpr int ES = DT == AR_BFLOAT16 ? 2 : 4;
    // fp32 accumulation holds 8 floats per 16-byte vector (bf16: one running
    // sum of 8 values; fp32: a block and a running sum of 4): at most
    // kStreamVpt vectors per thread stay in registers
    constexpr bool kAccOk = VPT <= kStreamVpt;
    constexpr int NA = kAccOk ? VPT : 1;
    const int lane = ct & 31;
    uint32_t g = 0;
    for (uint32_t it = blockIdx.x; it < a.n_items; it += gridDim.x) {
        const WorkItem w = a.items[it];
        const DevProg pg = a.progs[w.prog];
        const uint32_t nvec = (w.count * ES) >> 4;
        const int64_t off = w.elem * ES;
        uint4 res[VPT];
        if (pg.kind == PK_TREE) {
            if constexpr (TREES) {
                // bf16 trees on whole tiles drop the per-vector bounds test:
                // measured +6% on RH's reduce-scatter, +4% at P = 64 (fp32
                // trees gained nothing and keep one instantiation)
                constexpr bool kWholeTilePath = DT == AR_BFLOAT16;
                const bool ok = (kWholeTilePath && nvec == static_cast<uint32_t>(VPT * kConsumers))
                                    ? stream_tree<DT, OP, VPT, kWholeTilePath, TM>(a, sm, pg, g, off, nvec, ct, tstack)
                                    : stream_tree<DT, OP, VPT, false, TM>(a, sm, pg, g, off, nvec, ct, tstack);
                if (!ok) return;
            } else {
                atomicOr(a.status, kStatusBadProgram);
                return;
            }
        } else if (pg.kind == PK_ACC) {
            if (!kAccOk || TREES) {
                atomicOr(a.status, kStatusBadProgram);
                return;
            }
            AccStream<DT, OP> acc[NA];
            for (uint32_t i = 0; i < pg.n_in; ++i, ++g) {
                const uint32_t t = stream_acquire(a, sm, g);
                if (!t) return;
#pragma unroll
                for (int j = 0; j < NA; ++j) {
                    const uint32_t v = ct + j * kConsumers;
                    if (v < nvec) acc[j].feed(i, lds128(t + v * 16));
                }
                if (i + 1 < pg.n_in) {
                    stream_release(a, sm, g, lane);
                } else {
#pragma unroll
                    for (int j = 0; j < NA; ++j) res[j] = acc[j].finish(pg.n_in, avg_div(a, pg));
                    stream_finish<VPT>(a, sm, g, t, pg, off, nvec, ct, res);
                }
            }
        } else {
            const bool right = pg.kind == PK_CHAIN_R;
            for (uint32_t i = 0; i < pg.n_in; ++i, ++g) {
                const uint32_t t = stream_acquire(a, sm, g);
                if (!t) return;
                if (i == 0) {
#pragma unroll
                    for (int j = 0; j < VPT; ++j) {
                        const uint32_t v = ct + j * kConsumers;
                        if (v < nvec) res[j] = lds128(t + v * 16);
                    }
                } else if (right) {
#pragma unroll
                    for (int j = 0; j < VPT; ++j) {
                        const uint32_t v = ct + j * kConsumers;
                        if (v < nvec) res[j] = vop<DT, OP>(lds128(t + v * 16), res[j]);
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < VPT; ++j) {
                        const uint32_t v = ct + j * kConsumers;
                        if (v < nvec) res[j] = vop<DT, OP>(res[j], lds128(t + v * 16));
                    }
                }
                if (i + 1 < pg.n_in) {
                    stream_release(a, sm, g, lane);
                } else {
                    if (pg.flags & PF_AVG) {
#pragma unroll
                        for (int j = 0; j < VPT; ++j) res[j] = vdiv<DT>(res[j], static_cast<float>(a.P));
                    }
                    stream_finish<VPT>(a, sm, g, t, pg, off, nvec, ct, res);
                }
            }
        }
    }
}

// TM (tree instantiations): the tree stack in tensor memory; the first
// consumer warp allocates kTmemCols columns before the roles split and frees
// them after every consumer warp is done (a named barrier among them), on
// every path out of the consumer loop.
template <int DT, int OP, int VPT, bool TREES, bool TM = false>
__global__ void __launch_bounds__(kStreamThreads, 1) stream_kernel(const __grid_constant__ KernelArgs a) {
    extern __shared__ __align__(128) uint8_t smem[];
    constexpr int ES = DT == AR_BFLOAT16 ? 2 : 4;
    Stage sm;
    sm.full = smem_addr(smem);
    sm.empty = sm.full + 8 * a.stages;
    sm.ready = sm.empty + 8 * a.stages;
    sm.tiles = sm.full + kBarrierBytes;
    sm.stage_bytes = a.tile_bytes;
    // rank-streaming kernel: the tree stack's a.max_tmp tiles follow the stages
    sm.tmps = sm.tiles + a.stages * a.tile_bytes;
    if (threadIdx.x == 0) {
        for (int s = 0; s < a.stages; ++s) {
            mbar_init(sm.full + 8 * s, 1);
            mbar_init(sm.empty + 8 * s, kConsumerWarps);
            mbar_init(sm.ready + 8 * s, kConsumerWarps);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    const int warp = threadIdx.x >> 5;
    const uint32_t tslot = sm.full + kTmemAddrOffset;  // the allocated address, in the barrier area
    if constexpr (TM) {
        if (warp == kStreamLead) tmem_alloc(tslot, kTmemCols);
        tmem_fence_before();
    }
    __syncthreads();
    if constexpr (TM) tmem_fence_after();
    griddep_wait();
    griddep_launch_dependents();
    if (warp == 0) {
        stream_produce<ES>(a, sm);
        return;
    }
    if (warp == 1) {
        if (threadIdx.x == 32 && (a.flags & kArgTmaStore)) stream_store<ES>(a, sm);
        return;
    }
    uint32_t tstack = 0;
    if constexpr (TM) {
        // this warp's quarter of the lanes; the two consumer warps on a
        // quarter split its columns
        const uint32_t base = *reinterpret_cast<volatile uint32_t*>(smem + kTmemAddrOffset);
        tstack = base + ((32u * (warp & 3)) << 16) + (warp >= kStreamLead + 4 ? kTmemCols / 2 : 0u);
    }
    stream_consume<DT, OP, VPT, TREES, TM>(a, sm, threadIdx.x - 32 * kStreamLead, tstack);
    if constexpr (TM) {
        tmem_wait_st();
        tmem_fence_before();
        asm volatile("bar.sync 1, %0;" ::"r"(32 * kConsumerWarps) : "memory");
        if (warp == kStreamLead) {
            tmem_fence_after();
            tmem_dealloc(*reinterpret_cast<volatile uint32_t*>(smem + kTmemAddrOffset), kTmemCols);
        }
    }
}

// --------------------------------------------------------- element kernel

template <int DT>
__device__ __forceinline__ uint32_t ld_elem(const char* p) {
    if (DT == AR_BFLOAT16) return *reinterpret_cast<const uint16_t*>(p);
    return *reinterpret_cast<const uint32_t*>(p);
}

template <int DT>
__device__ __forceinline__ void st_elem(char* p, uint32_t v) {
    if (DT == AR_BFLOAT16)
        *reinterpret_cast<uint16_t*>(p) = static_cast<uint16_t>(v);
    else
        *reinterpret_cast<uint32_t*>(p) = v;
}

// a (+) b on one element (bf16 in the low half of the word)
template <int DT, int OP>
__device__ __forceinline__ uint32_t eop(uint32_t a, uint32_t b) {
    if (DT == AR_BFLOAT16) return wop<DT, OP>(a & 0xFFFFu, b & 0xFFFFu) & 0xFFFFu;
    return wop<DT, OP>(a, b);
}

// one element's AR_AVG division when div != 0
template <int DT>
__device__ __forceinline__ uint32_t ediv(uint32_t v, float div) {
    if (div == 0.f) return v;
    if (DT == AR_BFLOAT16) return wdiv<DT>(v & 0xFFFFu, div) & 0xFFFFu;
    return wdiv<DT>(v, div);
}

template <int DT, int OP>
__global__ void __launch_bounds__(kElemThreads) elementwise_kernel(const __grid_constant__ KernelArgs a) {
    extern __shared__ uint32_t vals[];  // [(max_in + max_tmp) rows][kElemThreads]
    constexpr int ES = DT == AR_BFLOAT16 ? 2 : 4;
    griddep_wait();
    griddep_launch_dependents();
    const WorkItem w = a.items[blockIdx.x];
    const DevProg pg = a.progs[w.prog];
    const int t = threadIdx.x;
    auto row = [&](uint32_t r) -> uint32_t& {
        return (r & REF_TMP) ? vals[(a.max_in + (r & 0x1FFu)) * kElemThreads + t] : vals[r * kElemThreads + t];
    };
    if (pg.kind == PK_TREE) {
        // a tree deeper than the stack (never emitted by the lowering) is
        // refused by every thread alike, before any barrier
        int sp = 0;
        for (uint32_t i = 0; i < pg.n_in; ++i) {
            if (++sp > kTreeDepth) {
                if (t == 0) atomicOr(a.status, kStatusBadProgram);
                return;
            }
            sp -= min(static_cast<int>((a.ins[pg.ins_off + (i >> 3)] >> (4 * (i & 7))) & 15u), sp - 1);
        }
    }
    // Blocks of up to 64 elements.  All threads load a block's inputs
    // together (value q is input q / cnt of element q % cnt, so a tiny item
    // with many inputs still has every thread loading), then each thread
    // evaluates the program for its element.
    for (uint32_t base = 0; base < w.count; base += kElemThreads) {
        const uint32_t cnt = min(static_cast<uint32_t>(kElemThreads), w.count - base);
        const uint32_t total = cnt * pg.n_in;
        uint32_t q = t;
        for (; q + 3 * kElemThreads < total; q += 4 * kElemThreads) {
            uint32_t v[4], slot[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const uint32_t qq = q + k * kElemThreads, i = qq / cnt, e = qq - i * cnt;
                v[k] = ld_elem<DT>(buf_addr(a, a.refs[pg.in_off + i]) + (w.elem + base + e) * ES);
                slot[k] = i * kElemThreads + e;
            }
#pragma unroll
            for (int k = 0; k < 4; ++k) vals[slot[k]] = v[k];
        }
        for (; q < total; q += kElemThreads) {
            const uint32_t i = q / cnt, e = q - i * cnt;
            vals[i * kElemThreads + e] = ld_elem<DT>(buf_addr(a, a.refs[pg.in_off + i]) + (w.elem + base + e) * ES);
        }
        __syncthreads();
        if (static_cast<uint32_t>(t) < cnt) {
            const int64_t off = (w.elem + base + t) * ES;
            if (pg.kind == PK_CHAIN_R || pg.kind == PK_CHAIN_L) {
                uint32_t acc = vals[t];
                for (uint32_t i = 1; i < pg.n_in; ++i) {
                    const uint32_t x = vals[i * kElemThreads + t];
                    acc = pg.kind == PK_CHAIN_R ? eop<DT, OP>(x, acc) : eop<DT, OP>(acc, x);
                }
                acc = ediv<DT>(acc, avg_div(a, pg));
                for (uint32_t o = 0; o < pg.n_out; ++o) st_elem<DT>(buf_addr(a, a.refs[pg.out_off + o]) + off, acc);
            } else if (pg.kind == PK_TREE) {
                // post-order on a small stack (local memory is fine on this path)
                uint32_t stk[kTreeDepth];
                int sp = 0;
                for (uint32_t i = 0; i < pg.n_in; ++i) {
                    stk[sp++] = vals[i * kElemThreads + t];  // depth checked above
                    for (uint32_t q = (a.ins[pg.ins_off + (i >> 3)] >> (4 * (i & 7))) & 15u; q > 0 && sp >= 2; --q, --sp)
                        stk[sp - 2] = eop<DT, OP>(stk[sp - 2], stk[sp - 1]);
                }
                const uint32_t res = ediv<DT>(stk[0], avg_div(a, pg));
                for (uint32_t o = 0; o < pg.n_out; ++o) st_elem<DT>(buf_addr(a, a.refs[pg.out_off + o]) + off, res);
            } else if (pg.kind == PK_ACC) {
                // the same order as the other kernels: the element rides in lane 0
                // of a vector (the other lanes carry zeros and are dropped)
                const uint4 r = acc_reduce<DT, OP>(pg.n_in, avg_div(a, pg), [&](uint32_t i) {
                    return make_uint4(vals[i * kElemThreads + t], 0u, 0u, 0u);
                });
                const uint32_t v = DT == AR_BFLOAT16 ? (r.x & 0xFFFFu) : r.x;
                for (uint32_t o = 0; o < pg.n_out; ++o) st_elem<DT>(buf_addr(a, a.refs[pg.out_off + o]) + off, v);
            } else {
                uint32_t acc = 0;
                for (uint32_t q = 0; q < pg.n_ins; ++q) {
                    const uint32_t wd = a.ins[pg.ins_off + q];
                    if ((wd >> 30) == INS_OP) {
                        const uint32_t ra = wd & 0x3FFu, rb = (wd >> 10) & 0x3FFu, rd = (wd >> 20) & 0x3FFu;
                        const uint32_t x = ra == REF_ACC ? acc : row(ra);
                        const uint32_t y = rb == REF_ACC ? acc : row(rb);
                        const uint32_t r = eop<DT, OP>(x, y);
                        if (rd == REF_ACC)
                            acc = r;
                        else
                            row(rd) = r;
                    } else {
                        const uint32_t rv = wd & 0x3FFu, id = (wd >> 10) & 0xFFFFu;
                        const float div = (wd >> 30) == INS_STORE_AVG ? static_cast<float>(a.P) : 0.f;
                        st_elem<DT>(buf_addr(a, id) + off, ediv<DT>(rv == REF_ACC ? acc : row(rv), div));
                    }
                }
            }
        }
        __syncthreads();  // the block's values are read before the next block's loads
    }
}

// --------------------------------------------------------- wait self-test

// One CTA waits on an mbarrier that nothing completes, gives up after ns
// nanoseconds the way every kernel's bounded wait does, records the same
// status bit and returns.
__global__ void wait_selftest_kernel(int* status, uint64_t ns) {
    __shared__ __align__(8) uint64_t bar;
    const uint32_t b = smem_addr(&bar);
    if (threadIdx.x == 0) {
        mbar_init(b, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    if (threadIdx.x == 0 && !mbar_wait_for(b, 0, ns)) atomicOr(status, kStatusWaitFull);
}

// ------------------------------------------------------- chain word kernel
//
// Chains (the ring's and the pipelined chain's programs) over passes too small
// to fill the GPU with rank tiles.  A thread takes 32-bit words at the same
// offset of every input buffer: k = kChainWordMaxIn / n_in word positions per
// round (every input of each), so it has kChainWordMaxIn loads in flight
// whatever P is, held in a register array indexed only by unrolled constants.
// It folds each position's words in the program's order and stores the result
// word to every output.  An item's buffer addresses are resolved once, into
// shared memory, by the whole CTA.  Plain (cached) loads and stores: these
// passes are small enough that their data may stay in L2 between calls.
__device__ __forceinline__ uint32_t ld32(const char* p) {
    uint32_t v;
    asm volatile("ld.global.b32 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}

__device__ __forceinline__ void st32(char* p, uint32_t v) {
    asm volatile("st.global.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

template <int DT, int OP, int M>
__global__ void __launch_bounds__(kChainWordThreads) chain_word_kernel(const __grid_constant__ KernelArgs a) {
    constexpr int ES = DT == AR_BFLOAT16 ? 2 : 4;
    constexpr int K = kChainWordMaxIn / M;  // word positions per thread per round
    __shared__ const char* src[M];
    __shared__ char* dst[kChainWordMaxIn];
    griddep_wait();
    griddep_launch_dependents();
    for (uint32_t it = blockIdx.x; it < a.n_items; it += gridDim.x) {
        const WorkItem w = a.items[it];
        const DevProg pg = a.progs[w.prog];
        if ((pg.kind != PK_CHAIN_R && pg.kind != PK_CHAIN_L) || pg.n_in < 1 || pg.n_in > M ||
            pg.n_out > kChainWordMaxIn) {
            if (threadIdx.x == 0) atomicOr(a.status, kStatusBadProgram);
            return;  // every thread alike, before any barrier of this item
        }
        const int64_t off = w.elem * ES;
        __syncthreads();  // the previous item's addresses are read no more
        for (uint32_t i = threadIdx.x; i < pg.n_in; i += blockDim.x) src[i] = buf_addr(a, a.refs[pg.in_off + i]) + off;
        for (uint32_t o = threadIdx.x; o < pg.n_out; o += blockDim.x) dst[o] = out_addr(a, pg, o) + off;
        __syncthreads();
        const uint32_t n = pg.n_in;
        const uint32_t nw = (w.count * ES) >> 2;
        const bool right = pg.kind == PK_CHAIN_R;
        const float div = avg_div(a, pg);
        for (uint32_t base = threadIdx.x; base < nw; base += K * blockDim.x) {
            uint32_t x[K][M];
#pragma unroll
            for (int i = 0; i < M; ++i)
#pragma unroll
                for (int j = 0; j < K; ++j) {
                    const uint32_t pos = base + j * blockDim.x;
                    if (i < n && pos < nw) x[j][i] = ld32(src[i] + 4 * pos);
                }
#pragma unroll
            for (int j = 0; j < K; ++j) {
                const uint32_t pos = base + j * blockDim.x;
                if (pos >= nw) break;
                uint32_t acc = x[j][0];
#pragma unroll
                for (int i = 1; i < M; ++i)
                    if (i < n) acc = right ? wop<DT, OP>(x[j][i], acc) : wop<DT, OP>(acc, x[j][i]);
                if (div != 0.f) acc = wdiv<DT>(acc, div);
                for (uint32_t o = 0; o < pg.n_out; ++o) st32(dst[o] + 4 * pos, acc);
            }
        }
    }
}

// ------------------------------------------------------------- copy kernel
//
// Fused passes that only copy (all-gathers: one input chunk, written to every
// other rank) move (P - 1) bytes out for each byte in, and what bounds them is
// how many stores the SMs keep in flight.  The rank-streaming kernel, one CTA
// of 10 warps per SM with TMA bulk stores, reached 90% of the copy peak on
// them.  Here a CTA of 256 threads takes one 16 KB item: each thread loads
// its AR_COPY_UNROLL 16-byte vectors (4 of them) before it stores them to
// every output, and the grid has a CTA per item, so that the hardware keeps
// every SM full of CTAs (64 registers: 4 resident per SM) as earlier ones
// finish.  Measured at 256 MiB per rank (P = 2 ... 16, 32 MiB at P = 64):
// a persistent grid of 8 CTAs per SM over 32 KB items 90-94% of the copy
// peak, 32 CTAs per SM 97-99%, a CTA per 32 KB item 98-100%, per 16 KB item
// 99.5-102% (above 1: the peak is a 1 : 1 copy, these passes mostly write);
// 8 KB items 80% at P = 2.  A CTA's threads share the item's addresses
// through shared memory.
#ifndef AR_COPY_UNROLL
#define AR_COPY_UNROLL 8
#endif

__device__ __forceinline__ uint4 ldg128_cs(const char* p) {
    uint4 v;
    asm volatile("ld.global.cs.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

template <int ES>
__global__ void __launch_bounds__(kCopyThreads) copy_kernel(const __grid_constant__ KernelArgs a) {
    constexpr int U = AR_COPY_UNROLL;
    __shared__ const char* src;
    __shared__ char* dst[AR_MAX_RANKS];
    griddep_wait();
    griddep_launch_dependents();
    for (uint32_t it = blockIdx.x; it < a.n_items; it += gridDim.x) {
        const WorkItem w = a.items[it];
        const DevProg pg = a.progs[w.prog];
        if ((pg.kind != PK_CHAIN_R && pg.kind != PK_CHAIN_L) || pg.n_in != 1 || pg.n_out > AR_MAX_RANKS ||
            (pg.flags & PF_AVG)) {
            if (threadIdx.x == 0) atomicOr(a.status, kStatusBadProgram);
            return;  // every thread alike, before any barrier of this item
        }
        const int64_t off = w.elem * ES;
        __syncthreads();  // the previous item's addresses are read no more
        if (threadIdx.x == 0) src = buf_addr(a, a.refs[pg.in_off]) + off;
        for (uint32_t o = threadIdx.x; o < pg.n_out; o += blockDim.x) dst[o] = out_addr(a, pg, o) + off;
        __syncthreads();
        const char* s = src;
        const uint32_t nv = (w.count * ES) >> 4;  // bulk items are whole 16-byte vectors
        for (uint32_t base = threadIdx.x; base < nv; base += U * blockDim.x) {
            uint4 v[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const uint32_t q = base + u * blockDim.x;
                if (q < nv) v[u] = ldg128_cs(s + 16ull * q);
            }
            for (uint32_t o = 0; o < pg.n_out; ++o) {
                char* d = dst[o];
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const uint32_t q = base + u * blockDim.x;
                    if (q < nv) stg128(d + 16ull * q, v[u]);
                }
            }
        }
    }
}

// ------------------------------------------------------- few-input kernel
//
// Fused passes of chains or fp32 accumulations of at most kFewMaxIn inputs
// (the ring's fused pass at P <= 16) on the copy kernel's grid shape: a CTA
// per 16 KB item, each thread loading its U 16-byte vectors of every input
// before it folds them in the program's order (a chain: a2's element op; an
// accumulation: the fp32 order of the other kernels; avg divided where the
// program says) and stores the result to every output.  Instantiations,
// every load of a thread in flight at once: up to 4 inputs with two vectors
// per thread (64 registers, four CTAs per SM), up to 8 with two (102
// registers, two CTAs per SM), up to 16 with one (110 registers).  (The
// 8-input one at P = 2 held too few loads in flight per SM: 77% of the copy
// peak against 100.5%.)
//
// The TREES instantiations (up to 4 leaves with two vectors per thread, 90
// registers; up to kFewTreeMaxIn with one, 80) run single trees too, with
// chains: the program's leaves in post-order with the combines that follow
// each (4 bits a leaf, as the rank-streaming kernel reads them), the top of
// the stack in registers and at most few_tree_stack(M) deeper entries in
// registers indexed by unrolled selects (the stack pointer is the same in
// every thread).
#ifndef AR_FEW_TREE_UNROLL
#define AR_FEW_TREE_UNROLL 1
#endif
template <int DT, int OP, int M, int U, bool TREES>
__global__ void __launch_bounds__(kCopyThreads) few_kernel(const __grid_constant__ KernelArgs a) {
    constexpr int ES = DT == AR_BFLOAT16 ? 2 : 4;
    constexpr int S = few_tree_stack(M);
    __shared__ const char* src[M];
    __shared__ char* dst[AR_MAX_RANKS];
    __shared__ uint32_t counts[(M + 7) / 8];
    griddep_wait();
    griddep_launch_dependents();
    for (uint32_t it = blockIdx.x; it < a.n_items; it += gridDim.x) {
        const WorkItem w = a.items[it];
        const DevProg pg = a.progs[w.prog];
        const bool kind_ok = pg.kind == PK_CHAIN_R || pg.kind == PK_CHAIN_L ||
                             (TREES ? pg.kind == PK_TREE && pg.n_tmp <= S : pg.kind == PK_ACC);
        if (!kind_ok || pg.n_in < 1 || pg.n_in > M || pg.n_out > AR_MAX_RANKS) {
            if (threadIdx.x == 0) atomicOr(a.status, kStatusBadProgram);
            return;  // every thread alike, before any barrier of this item
        }
        const int64_t off = w.elem * ES;
        __syncthreads();  // the previous item's addresses are read no more
        for (uint32_t i = threadIdx.x; i < pg.n_in; i += blockDim.x) src[i] = buf_addr(a, a.refs[pg.in_off + i]) + off;
        for (uint32_t o = threadIdx.x; o < pg.n_out; o += blockDim.x) dst[o] = out_addr(a, pg, o) + off;
        if (TREES && pg.kind == PK_TREE && threadIdx.x < (pg.n_in + 7) / 8) counts[threadIdx.x] = a.ins[pg.ins_off + threadIdx.x];
        __syncthreads();
        const uint32_t n = pg.n_in;
        const bool right = pg.kind == PK_CHAIN_R;
        const float div = avg_div(a, pg);
        const uint32_t nv = (w.count * ES) >> 4;  // bulk items are whole 16-byte vectors
        for (uint32_t base = threadIdx.x; base < nv; base += U * blockDim.x) {
            uint4 x[M][U];
#pragma unroll
            for (int i = 0; i < M; ++i)
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const uint32_t q = base + u * blockDim.x;
                    if (i < static_cast<int>(n) && q < nv) x[i][u] = ldg128_cs(src[i] + 16ull * q);
                }
            if (TREES && pg.kind == PK_TREE) {
                uint4 acc[U], st[S][U];
                uint32_t sp = 0;  // stack entries, the top one in acc
#pragma unroll
                for (int i = 0; i < M; ++i) {
                    if (i < static_cast<int>(n)) {
                        uint32_t c = (counts[i >> 3] >> (4 * (i & 7))) & 15u;
                        if (sp == 0 || c == 0) {
#pragma unroll
                            for (int d = 0; d < S; ++d)
                                if (d + 1 == static_cast<int>(sp))
#pragma unroll
                                    for (int u = 0; u < U; ++u) st[d][u] = acc[u];
#pragma unroll
                            for (int u = 0; u < U; ++u) acc[u] = x[i][u];
                            ++sp;
                        } else {
#pragma unroll
                            for (int u = 0; u < U; ++u) acc[u] = vop<DT, OP>(acc[u], x[i][u]);
                            --c;
                        }
                        for (; c > 0; --c, --sp) {
#pragma unroll
                            for (int d = 0; d < S; ++d)
                                if (d + 2 == static_cast<int>(sp))
#pragma unroll
                                    for (int u = 0; u < U; ++u) acc[u] = vop<DT, OP>(st[d][u], acc[u]);
                        }
                    }
                }
#pragma unroll
                for (int u = 0; u < U; ++u) x[0][u] = div != 0.f ? vdiv<DT>(acc[u], div) : acc[u];
            } else if (pg.kind == PK_ACC) {
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    AccStream<DT, OP> s;
#pragma unroll
                    for (int i = 0; i < M; ++i)
                        if (i < static_cast<int>(n)) s.feed(i, x[i][u]);
                    x[0][u] = s.finish(n, div);
                }
            } else {
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    uint4 acc = x[0][u];
#pragma unroll
                    for (int i = 1; i < M; ++i)
                        if (i < static_cast<int>(n)) acc = right ? vop<DT, OP>(x[i][u], acc) : vop<DT, OP>(acc, x[i][u]);
                    x[0][u] = div != 0.f ? vdiv<DT>(acc, div) : acc;
                }
            }
            for (uint32_t o = 0; o < pg.n_out; ++o) {
                char* d = dst[o];
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const uint32_t q = base + u * blockDim.x;
                    if (q < nv) stg128(d + 16ull * q, x[0][u]);
                }
            }
        }
    }
}

// Chains and fp32 accumulations of more than kFewMaxIn inputs (up to
// AR_MAX_RANKS) on the same grid shape: a thread folds its vector of each
// item in groups of AR_FEW_LONG_GROUP inputs, every load of a group in
// flight at once, in the program's order across the groups; registers
// capped for AR_FEW_LONG_MIN_CTAS CTAs per SM.  Measured at 64-256 MiB per
// rank, P = 32 / 64, fp32 / bf16, faithful / fp32-accumulate: groups of 8
// with three CTAs per SM (80 registers) 98.5-100.8% of the copy peak,
// groups of 16 with two (128) within a point of it, groups of 16 with one
// (142 registers) 91-95%, the rank-streaming kernel 89.6-96.8%.
#ifndef AR_FEW_LONG_GROUP
#define AR_FEW_LONG_GROUP 8
#endif
#ifndef AR_FEW_LONG_MIN_CTAS
#define AR_FEW_LONG_MIN_CTAS 3
#endif
template <int DT, int OP>
__global__ void __launch_bounds__(kCopyThreads, AR_FEW_LONG_MIN_CTAS) few_long_kernel(const __grid_constant__ KernelArgs a) {
    constexpr int ES = DT == AR_BFLOAT16 ? 2 : 4;
    constexpr int G = AR_FEW_LONG_GROUP;
    __shared__ const char* src[AR_MAX_RANKS];
    __shared__ char* dst[AR_MAX_RANKS];
    griddep_wait();
    griddep_launch_dependents();
    for (uint32_t it = blockIdx.x; it < a.n_items; it += gridDim.x) {
        const WorkItem w = a.items[it];
        const DevProg pg = a.progs[w.prog];
        if ((pg.kind != PK_CHAIN_R && pg.kind != PK_CHAIN_L && pg.kind != PK_ACC) || pg.n_in < 1 ||
            pg.n_in > AR_MAX_RANKS || pg.n_out > AR_MAX_RANKS) {
            if (threadIdx.x == 0) atomicOr(a.status, kStatusBadProgram);
            return;  // every thread alike, before any barrier of this item
        }
        const int64_t off = w.elem * ES;
        __syncthreads();  // the previous item's addresses are read no more
        for (uint32_t i = threadIdx.x; i < pg.n_in; i += blockDim.x) src[i] = buf_addr(a, a.refs[pg.in_off + i]) + off;
        for (uint32_t o = threadIdx.x; o < pg.n_out; o += blockDim.x) dst[o] = out_addr(a, pg, o) + off;
        __syncthreads();
        const uint32_t n = pg.n_in;
        const bool right = pg.kind == PK_CHAIN_R, accumulate = pg.kind == PK_ACC;
        const float div = avg_div(a, pg);
        const uint32_t nv = (w.count * ES) >> 4;  // bulk items are whole 16-byte vectors
        for (uint32_t q = threadIdx.x; q < nv; q += blockDim.x) {
            AccStream<DT, OP> s;
            uint4 acc;
            for (uint32_t g0 = 0; g0 < n; g0 += G) {
                uint4 x[G];
#pragma unroll
                for (int i = 0; i < G; ++i)
                    if (g0 + i < n) x[i] = ldg128_cs(src[g0 + i] + 16ull * q);
#pragma unroll
                for (int i = 0; i < G; ++i) {
                    if (g0 + i >= n) break;
                    if (accumulate)
                        s.feed(g0 + i, x[i]);
                    else if (g0 + i == 0)
                        acc = x[i];
                    else
                        acc = right ? vop<DT, OP>(x[i], acc) : vop<DT, OP>(acc, x[i]);
                }
            }
            const uint4 r = accumulate ? s.finish(n, div) : (div != 0.f ? vdiv<DT>(acc, div) : acc);
            for (uint32_t o = 0; o < pg.n_out; ++o) stg128(dst[o] + 16ull * q, r);
        }
    }
}

// ----------------------------------------------------------------- dispatch

using KernelFn = void (*)(KernelArgs);

enum Which {
    K_STAGED = 0, K_STREAM = 1, K_ELEM = 3, K_STREAM_TREE = 4, K_STREAM_TREE_WIDE = 5, K_STREAM_MID = 6,
    K_CHAIN_WORD = 7, K_CHAIN_WORD8 = 8, K_CHAIN_WORD16 = 9, K_STREAM_TREE_TMEM = 10, K_FEW8 = 11, K_FEW16 = 12,
    K_FEW4 = 13, K_FEW_TREE8 = 14, K_FEW_TREE4 = 15, K_FEW_LONG = 16
};
constexpr int kWhich[] = {K_STAGED,     K_STREAM,     K_ELEM,        K_STREAM_TREE,  K_STREAM_TREE_WIDE,
                          K_STREAM_MID, K_CHAIN_WORD, K_CHAIN_WORD8, K_CHAIN_WORD16, K_STREAM_TREE_TMEM,
                          K_FEW8,       K_FEW16,      K_FEW4,        K_FEW_TREE8,    K_FEW_TREE4,
                          K_FEW_LONG};

template <int DT, int OP>
KernelFn table(int which) {
    if (which == K_STAGED) return staged_kernel<DT, OP>;
    if (which == K_STREAM) return stream_kernel<DT, OP, kStreamVpt, false>;
    // bf16 fp32 accumulation on 24 KB tiles: 48 accumulators per thread stay
    // in registers (with 64, the 32 KB tile's kernel spills)
    if constexpr (DT == AR_BFLOAT16)
        if (which == K_STREAM_MID) return stream_kernel<DT, OP, kStreamVptTree, false>;
    if (which == K_STREAM_MID) return nullptr;
    if (which == K_CHAIN_WORD8) return chain_word_kernel<DT, OP, 8>;
    if (which == K_CHAIN_WORD16) return chain_word_kernel<DT, OP, 16>;
    if (which == K_CHAIN_WORD) return chain_word_kernel<DT, OP, kChainWordMaxIn>;
    if (which == K_FEW4) return few_kernel<DT, OP, 4, 2, false>;
    if (which == K_FEW8) return few_kernel<DT, OP, 8, 2, false>;
    if (which == K_FEW16) return few_kernel<DT, OP, kFewMaxIn, 1, false>;
    if (which == K_FEW_TREE4) return few_kernel<DT, OP, 4, 2, true>;
    if (which == K_FEW_LONG) return few_long_kernel<DT, OP>;
    if (which == K_FEW_TREE8) return few_kernel<DT, OP, 8, AR_FEW_TREE_UNROLL, true>;
    if (which == K_STREAM_TREE) return stream_kernel<DT, OP, kStreamVptTree, true>;
    if (which == K_STREAM_TREE_WIDE) return stream_kernel<DT, OP, kStreamVpt, true>;
    if (which == K_STREAM_TREE_TMEM) return stream_kernel<DT, OP, kStreamVpt, true, true>;
    return elementwise_kernel<DT, OP>;
}

template <int DT>
KernelFn pick(int op, int which) {
    switch (op) {
        case AR_SUM:
        case AR_AVG: return table<DT, AR_SUM>(which);  // AVG: the sum, divided where it completes
        case AR_PROD: return table<DT, AR_PROD>(which);
        case AR_MAX: return table<DT, AR_MAX>(which);
        default: return table<DT, AR_MIN>(which);
    }
}

KernelFn kernel_for(int dtype, int op, int which) {
    switch (dtype) {
        case AR_INT32: return pick<AR_INT32>(op, which);
        case AR_FLOAT32: return pick<AR_FLOAT32>(op, which);
        default: return pick<AR_BFLOAT16>(op, which);
    }
}

}  // namespace

cudaError_t launch_dependent(const void* f, int grid, int block, int smem, cudaStream_t st, const KernelArgs& a) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(static_cast<unsigned>(block));
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = AR_PDL;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    void* args[] = {const_cast<KernelArgs*>(&a)};
    return cudaLaunchKernelExC(&cfg, f, args);
}

cudaError_t launch_wait_selftest(int* status, uint64_t ns, cudaStream_t st) {
    wait_selftest_kernel<<<1, 32, 0, st>>>(status, ns);
    return cudaGetLastError();
}

cudaError_t prepare_kernels(int dtype, int op) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    int optin = 0;
    e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (e != cudaSuccess) return e;
    for (int which : kWhich) {
        KernelFn f = kernel_for(dtype, op, which);
        // (the chain word and few-input kernels have static shared memory only)
        if (!f || which == K_CHAIN_WORD || which == K_CHAIN_WORD8 || which == K_CHAIN_WORD16 || which == K_FEW4 ||
            which == K_FEW8 || which == K_FEW16 || which == K_FEW_TREE8 || which == K_FEW_TREE4 ||
            which == K_FEW_LONG)
            continue;
        e = cudaFuncSetAttribute(reinterpret_cast<const void*>(f), cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 optin);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

cudaError_t launch_staged(int dtype, int op, const KernelArgs& a, int grid, int smem, cudaStream_t st) {
    KernelFn f = kernel_for(dtype, op, K_STAGED);
    return launch_dependent(reinterpret_cast<const void*>(f), grid, kStagedThreads, smem, st, a);
}

cudaError_t launch_stream(int dtype, int op, const KernelArgs& a, int grid, int smem, cudaStream_t st) {
    // the rank tile fixes the vectors per consumer thread
    const int which = (a.flags & kArgTrees)
                          ? (a.tile_bytes == kStreamTileTree    ? K_STREAM_TREE
                             : a.tile_bytes == kStreamTileBytes && (a.flags & kArgTmemStack) ? K_STREAM_TREE_TMEM
                             : a.tile_bytes == kStreamTileBytes ? K_STREAM_TREE_WIDE
                                                                : -1)
                      : a.tile_bytes == kStreamTileBytes  ? K_STREAM
                      : a.tile_bytes == kStreamTileTree   ? K_STREAM_MID
                                                          : -1;
    if (which < 0) return cudaErrorInvalidValue;
    if (!kernel_for(dtype, op, which)) return cudaErrorInvalidValue;
    if (a.stages < 1 || a.stages > 32 || 24 * a.stages > kBarrierBytes) return cudaErrorInvalidValue;
    return launch_dependent(reinterpret_cast<const void*>(kernel_for(dtype, op, which)), grid, kStreamThreads, smem,
                            st, a);
}

cudaError_t launch_chain_words(int dtype, int op, const KernelArgs& a, int max_in, int grid, cudaStream_t st) {
    const int which = max_in <= 8 ? K_CHAIN_WORD8 : max_in <= 16 ? K_CHAIN_WORD16 : K_CHAIN_WORD;
    KernelFn f = kernel_for(dtype, op, which);
    return launch_dependent(reinterpret_cast<const void*>(f), grid, kChainWordThreads, 0, st, a);
}

cudaError_t launch_few(int dtype, int op, const KernelArgs& a, int max_in, bool trees, int grid, cudaStream_t st) {
    KernelFn f = kernel_for(dtype, op,
                            trees ? (max_in <= 4 ? K_FEW_TREE4 : K_FEW_TREE8)
                                  : (max_in <= 4   ? K_FEW4
                                     : max_in <= 8 ? K_FEW8
                                     : max_in <= kFewMaxIn ? K_FEW16
                                                           : K_FEW_LONG));
    return launch_dependent(reinterpret_cast<const void*>(f), grid, kCopyThreads, 0, st, a);
}

cudaError_t launch_copies(int dtype, const KernelArgs& a, int grid, cudaStream_t st) {
    const void* f = dtype == AR_BFLOAT16 ? reinterpret_cast<const void*>(copy_kernel<2>)
                                         : reinterpret_cast<const void*>(copy_kernel<4>);
    return launch_dependent(f, grid, kCopyThreads, 0, st, a);
}

cudaError_t launch_elementwise(int dtype, int op, const KernelArgs& a, int smem, cudaStream_t st) {
    KernelFn f = kernel_for(dtype, op, K_ELEM);
    return launch_dependent(reinterpret_cast<const void*>(f), static_cast<int>(a.n_items), kElemThreads, smem, st, a);
}

}  // namespace ar
