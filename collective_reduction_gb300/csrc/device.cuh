// Device code shared by the engine's compiled kernels (kernels.cu) and the
// DAG kernels it compiles at run time for a plan: element arithmetic, memory
// and mbarrier helpers, and the staged kernel's producer / consumer loop.
// Compiles under nvcc and NVRTC (no host headers under NVRTC).
#pragma once

#include "kargs.hpp"

// Launch kernels as programmatic dependents of their predecessor (1) or
// plainly stream-ordered (0); the host side reads the same macro.
#ifndef AR_PDL
#define AR_PDL 1
#endif

namespace ar {
namespace {


constexpr uint64_t kWaitNs = 2000000000ull;  // bounded waits give up after 2 s
constexpr int kVpt = kStagedVpt;             // 16-byte vectors per consumer thread per item
constexpr int kConsumers = 32 * kConsumerWarps;

// ---------------------------------------------------------------- arithmetic

template <int OP>
__device__ __forceinline__ float fop(float a, float b) {
    if (OP == AR_SUM) return __fadd_rn(a, b);
    if (OP == AR_PROD) return __fmul_rn(a, b);
    if (OP == AR_MAX) return a > b ? a : b;
    return a < b ? a : b;
}

template <int OP>
__device__ __forceinline__ int32_t iop(int32_t a, int32_t b) {
    if (OP == AR_SUM) return static_cast<int32_t>(static_cast<uint32_t>(a) + static_cast<uint32_t>(b));
    if (OP == AR_PROD) return static_cast<int32_t>(static_cast<uint32_t>(a) * static_cast<uint32_t>(b));
    if (OP == AR_MAX) return a > b ? a : b;
    return a < b ? a : b;
}

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
// two fp32 values rounded to bf16 (nearest even) and packed, lo in bits 0..15
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    uint32_t d;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
    return d;
}

// Two bf16 sums (products) in one instruction, each the exact result rounded
// once to bf16, nearest even, subnormals kept.  That is bit for bit the
// element op's definition (computed in fp32, then rounded to bf16): a
// result rounded to nearest in a format of p' >= 2p + 2 significand bits and
// then to nearest in p bits equals the direct rounding for +, -, x, / and
// square root (Figueroa, "When is double rounding innocuous?", 1995), and
// fp32 carries 24 >= 2 * 8 + 2 bits over the same exponent range as bf16.
__device__ __forceinline__ uint32_t add_bf16x2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("add.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
__device__ __forceinline__ uint32_t mul_bf16x2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// bf16 max (min) on two pairs: per element a > b ? a : b (a < b ? a : b),
// the comparison one ordered bf16x2 compare, like the fp32 one: false when
// either value is NaN, +0 and -0 equal, subnormals compared exactly.
template <int OP>
__device__ __forceinline__ uint32_t select_bf16x2(uint32_t a, uint32_t b) {
    uint32_t lo, hi;
    if (OP == AR_MAX)
        asm("{\n\t.reg .pred p, q;\n\tsetp.gt.bf16x2 p|q, %2, %3;\n\t"
            "selp.b32 %0, %2, %3, p;\n\tselp.b32 %1, %2, %3, q;\n\t}"
            : "=r"(lo), "=r"(hi) : "r"(a), "r"(b));
    else
        asm("{\n\t.reg .pred p, q;\n\tsetp.lt.bf16x2 p|q, %2, %3;\n\t"
            "selp.b32 %0, %2, %3, p;\n\tselp.b32 %1, %2, %3, q;\n\t}"
            : "=r"(lo), "=r"(hi) : "r"(a), "r"(b));
    return (lo & 0xFFFFu) | (hi & 0xFFFF0000u);
}

// a (+) b on one 32-bit word: one int32 / fp32 element or two bf16 elements
template <int DT, int OP>
__device__ __forceinline__ uint32_t wop(uint32_t a, uint32_t b) {
    if (DT == AR_INT32) return static_cast<uint32_t>(iop<OP>(static_cast<int32_t>(a), static_cast<int32_t>(b)));
    if (DT == AR_FLOAT32) return __float_as_uint(fop<OP>(__uint_as_float(a), __uint_as_float(b)));
    if (OP == AR_SUM) return add_bf16x2(a, b);
    if (OP == AR_PROD) return mul_bf16x2(a, b);
    return select_bf16x2<OP>(a, b);
}

template <int DT, int OP>
__device__ __forceinline__ uint4 vop(uint4 a, uint4 b) {
    return make_uint4(wop<DT, OP>(a.x, b.x), wop<DT, OP>(a.y, b.y), wop<DT, OP>(a.z, b.z),
                      wop<DT, OP>(a.w, b.w));
}

// x / d, rounded to nearest even, for d the rank count (a positive integer).
// When d is a power of two its reciprocal is exact, and x * (1 / d) is the
// same real number as x / d, so rounding it once gives the same bits,
// subnormal results included: one multiply instead of a division.
__device__ __forceinline__ float div_rank_count(float x, float d) {
    const uint32_t b = __float_as_uint(d);
    if ((b & 0x7FFFFFu) == 0u) return __fmul_rn(x, __uint_as_float((254u - (b >> 23)) << 23));
    return __fdiv_rn(x, d);
}

// AR_AVG: a complete sum divided by the rank count d (IEEE division, round to
// nearest even; bf16 values divided in fp32 and rounded back to bf16).
template <int DT>
__device__ __forceinline__ uint32_t wdiv(uint32_t w, float d) {
    if (DT == AR_FLOAT32) return __float_as_uint(div_rank_count(__uint_as_float(w), d));
    if (DT == AR_BFLOAT16) return pack_bf16x2(div_rank_count(bf_lo(w), d), div_rank_count(bf_hi(w), d));
    return w;  // int32 has no average (refused when the plan is made)
}

template <int DT>
__device__ __forceinline__ uint4 vdiv(uint4 v, float d) {
    return make_uint4(wdiv<DT>(v.x, d), wdiv<DT>(v.y, d), wdiv<DT>(v.z, d), wdiv<DT>(v.w, d));
}

// Accumulator of the FP32ACC order: int32 stays int32 (exact in any order),
// fp32 and bf16 accumulate in fp32 and round once.
template <int DT>
struct Acc {
    static constexpr int W = DT == AR_BFLOAT16 ? 8 : 4;
    float f[W];
};
template <>
struct Acc<AR_INT32> {
    static constexpr int W = 4;
    int32_t i[4];
};

template <int DT>
__device__ __forceinline__ void acc_widen(Acc<DT>& x, uint4 v) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    if constexpr (DT == AR_INT32) {
#pragma unroll
        for (int q = 0; q < 4; ++q) x.i[q] = static_cast<int32_t>(w[q]);
    } else if constexpr (DT == AR_FLOAT32) {
#pragma unroll
        for (int q = 0; q < 4; ++q) x.f[q] = __uint_as_float(w[q]);
    } else {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            x.f[2 * q] = bf_lo(w[q]);
            x.f[2 * q + 1] = bf_hi(w[q]);
        }
    }
}

template <int DT, int OP>
__device__ __forceinline__ void acc_combine(Acc<DT>& x, const Acc<DT>& y) {
    if constexpr (DT == AR_INT32) {
#pragma unroll
        for (int q = 0; q < 4; ++q) x.i[q] = iop<OP>(x.i[q], y.i[q]);
    } else {
#pragma unroll
        for (int q = 0; q < Acc<DT>::W; ++q) x.f[q] = fop<OP>(x.f[q], y.f[q]);
    }
}

// AR_AVG on the fp32 accumulator, before the one rounding to the dtype
template <int DT>
__device__ __forceinline__ void acc_div(Acc<DT>& x, float d) {
    if constexpr (DT != AR_INT32) {
#pragma unroll
        for (int q = 0; q < Acc<DT>::W; ++q) x.f[q] = __fdiv_rn(x.f[q], d);
    }
}

template <int DT>
__device__ __forceinline__ uint4 acc_narrow(const Acc<DT>& x) {
    if constexpr (DT == AR_INT32)
        return make_uint4(static_cast<uint32_t>(x.i[0]), static_cast<uint32_t>(x.i[1]),
                          static_cast<uint32_t>(x.i[2]), static_cast<uint32_t>(x.i[3]));
    else if constexpr (DT == AR_FLOAT32)
        return make_uint4(__float_as_uint(x.f[0]), __float_as_uint(x.f[1]), __float_as_uint(x.f[2]),
                          __float_as_uint(x.f[3]));
    else
        return make_uint4(pack_bf16x2(x.f[0], x.f[1]), pack_bf16x2(x.f[2], x.f[3]), pack_bf16x2(x.f[4], x.f[5]),
                          pack_bf16x2(x.f[6], x.f[7]));
}

// FP32ACC order over inputs 0..n-1 (the kernels' own fixed order, identical
// in every kernel and for every rank).  fp32 and int32: blocks of 8
// consecutive inputs are each folded left to right, then the block results
// are folded left to right.  bf16: one fp32 running sum folded left to right
// over all inputs (its rounding error, at most (n - 1) fp32 half-units of
// the running magnitudes, stays far below the one final rounding to bf16,
// and one accumulator per value keeps a 32 KB rank tile in registers).
// fp32 / bf16 round once at the end (an AR_AVG sum divided by div first;
// div = 0 for the other ops).  Inputs are fed one at a time, so the order
// can be followed while inputs stream in.
template <int DT, int OP>
struct AccStream {
    static constexpr bool kBlocks = DT != AR_BFLOAT16;
    Acc<DT> acc, blk;
    __device__ __forceinline__ void feed(uint32_t i, uint4 x) {
        Acc<DT> w;
        acc_widen<DT>(w, x);
        if constexpr (!kBlocks) {
            if (i == 0)
                acc = w;
            else
                acc_combine<DT, OP>(acc, w);
            return;
        }
        if ((i & 7u) == 0)
            blk = w;
        else
            acc_combine<DT, OP>(blk, w);
        if ((i & 7u) == 7u) {
            if (i == 7u)
                acc = blk;
            else
                acc_combine<DT, OP>(acc, blk);
        }
    }
    __device__ __forceinline__ uint4 finish(uint32_t n, float div) {
        if (kBlocks && (n & 7u)) {
            if (n < 8u)
                acc = blk;
            else
                acc_combine<DT, OP>(acc, blk);
        }
        if (div != 0.f) acc_div<DT>(acc, div);
        return acc_narrow<DT>(acc);
    }
};

template <int DT, int OP, class Load>
__device__ __forceinline__ uint4 acc_reduce(uint32_t n, float div, Load load) {
    AccStream<DT, OP> s;
    for (uint32_t i = 0; i < n; ++i) s.feed(i, load(i));
    return s.finish(n, div);
}

// The divisor of a program's AR_AVG results, 0 when it stores plain results.
__device__ __forceinline__ float avg_div(const KernelArgs& a, const DevProg& pg) {
    return (pg.flags & PF_AVG) ? static_cast<float>(a.P) : 0.f;
}

// ------------------------------------------------------------- memory access

__device__ __forceinline__ char* buf_addr(const KernelArgs& a, uint32_t id) {
    const uint32_t slot = id >> 6, rank = id & 63u;
    if (slot == 0) return static_cast<char*>(a.bufs[rank]);
    return a.scratch + (static_cast<uint64_t>(slot - 1) * a.P + rank) * a.slot_stride;
}

__device__ __forceinline__ char* out_addr(const KernelArgs& a, const DevProg& pg, uint32_t o) {
    if (pg.flags & PF_OUT_ALL) return static_cast<char*>(a.bufs[o]);
    return buf_addr(a, a.refs[pg.out_off + o]);
}

// 32-bit global accesses of the run-time compiled word kernel: each value is
// read once and its slot written once by the same thread (streaming hints)
__device__ __forceinline__ uint32_t ldg32(const char* p) {
    uint32_t v;
    asm volatile("ld.global.cs.b32 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}

__device__ __forceinline__ void stg32(char* p, uint32_t v) {
    asm volatile("st.global.cs.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// 4-byte asynchronous global -> shared copies of this thread (the word
// kernel's prefetch), grouped; wait_group<N> returns once at most N of this
// thread's groups are still in flight, their data visible to the thread.
__device__ __forceinline__ void cp_async4(uint32_t dst, const char* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr));
    return v;
}

__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
    return v;
}

__device__ __forceinline__ void sts128(uint32_t addr, uint4 v) {
    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z),
                 "r"(v.w)
                 : "memory");
}

#ifndef AR_STORE_CS
#define AR_STORE_CS 1
#endif

// results are never re-read by the kernel: streaming (evict-first) stores
__device__ __forceinline__ void stg128(char* p, uint4 v) {
    if (AR_STORE_CS)
        asm volatile("st.global.cs.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
                     "r"(v.w)
                     : "memory");
    else
        asm volatile("st.global.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
                     "r"(v.w)
                     : "memory");
}

__device__ __forceinline__ uint64_t globaltimer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ------------------------------------------------------ tensor memory (TMEM)
//
// The rank-streaming kernel's deep-tree instantiation keeps its stack in the
// SM's tensor memory (256 KB: 128 lanes x 512 columns of 32 bits) instead of
// shared memory, which then holds only pipeline stages.  One warp allocates
// the columns (the address goes to shared memory for the others) and frees
// them once every user is done; a warp reaches the 32 lanes of its quarter
// (warp id mod 4), each thread its own lane.
__device__ __forceinline__ void tmem_alloc(uint32_t smem_dst, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_dst), "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tmem_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tmem_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// this thread's 8 x 16 bytes to 32 consecutive columns of its lane (the
// whole warp executes it)
__device__ __forceinline__ void tmem_store32(uint32_t taddr, const uint4 (&v)[8]) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr), "r"(v[0].x), "r"(v[0].y), "r"(v[0].z), "r"(v[0].w), "r"(v[1].x), "r"(v[1].y), "r"(v[1].z), "r"(v[1].w), "r"(v[2].x), "r"(v[2].y), "r"(v[2].z), "r"(v[2].w), "r"(v[3].x), "r"(v[3].y), "r"(v[3].z), "r"(v[3].w), "r"(v[4].x), "r"(v[4].y), "r"(v[4].z), "r"(v[4].w), "r"(v[5].x), "r"(v[5].y), "r"(v[5].z), "r"(v[5].w), "r"(v[6].x), "r"(v[6].y), "r"(v[6].z), "r"(v[6].w), "r"(v[7].x), "r"(v[7].y), "r"(v[7].z), "r"(v[7].w) : "memory");
}

// ... and back; waits for the warp's earlier stores and for this load
__device__ __forceinline__ void tmem_load32(uint32_t taddr, uint4 (&v)[8]) {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(v[0].x), "=r"(v[0].y), "=r"(v[0].z), "=r"(v[0].w), "=r"(v[1].x), "=r"(v[1].y), "=r"(v[1].z), "=r"(v[1].w), "=r"(v[2].x), "=r"(v[2].y), "=r"(v[2].z), "=r"(v[2].w), "=r"(v[3].x), "=r"(v[3].y), "=r"(v[3].z), "=r"(v[3].w), "=r"(v[4].x), "=r"(v[4].y), "=r"(v[4].z), "=r"(v[4].w), "=r"(v[5].x), "=r"(v[5].y), "=r"(v[5].z), "=r"(v[5].w), "=r"(v[6].x), "=r"(v[6].y), "=r"(v[6].z), "=r"(v[6].w), "=r"(v[7].x), "=r"(v[7].y), "=r"(v[7].z), "=r"(v[7].w)
        : "r"(taddr)
        : "memory");
}

__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// ------------------------------------------------------ dependent launches
//
// The engine launches its kernels with programmatic stream serialization: a
// launch that follows another kernel in the stream may start (CTA launch,
// barrier setup) while that kernel finishes.  A kernel touches global memory
// only after griddep_wait, which returns once the preceding grid has
// completed and its writes are visible (at once when there is none), and
// lets its successor start early with griddep_launch_dependents, which takes
// effect only when every CTA of the grid has issued it (so all of them are
// resident) or exited.
__device__ __forceinline__ void griddep_wait() {
#if AR_PDL
    asm volatile("griddepcontrol.wait;" ::: "memory");
#endif
}

__device__ __forceinline__ void griddep_launch_dependents() {
#if AR_PDL
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
#endif
}

// ------------------------------------------------------------------ mbarrier

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Waits for the phase of the given parity; false after ns nanoseconds.
__device__ __noinline__ bool mbar_wait_for(uint32_t bar, uint32_t parity, uint64_t ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer();
    for (;;) {
        for (int i = 0; i < 32; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (globaltimer() - t0 > ns) return false;
    }
}

// The kernels' wait: false after kWaitNs.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) { return mbar_wait_for(bar, parity, kWaitNs); }

// loads are read once: ask L2 to evict them first
#ifndef AR_L2_EVICT_FIRST
#define AR_L2_EVICT_FIRST 1
#endif

__device__ __forceinline__ uint64_t evict_first_policy() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar,
                                          uint64_t policy) {
    if (AR_L2_EVICT_FIRST) {
        asm volatile(
            "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], "
            "%4;" ::"r"(dst),
            "l"(src), "r"(bytes), "r"(bar), "l"(policy)
            : "memory");
    } else {
        asm volatile(
            "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
            "l"(src), "r"(bytes), "r"(bar)
            : "memory");
    }
}

// ------------------------------------------------------------ staged kernel

struct Stage {
    uint32_t full, empty;  // mbarrier arrays (shared addresses)
    uint32_t ready;        // rank-streaming kernel: per stage, an item's result is in it
    uint32_t tiles;        // stage 0 tiles
    uint32_t tmps;         // temporaries
    uint32_t stage_bytes;
};

// Items with more inputs than this take the warp-wide staged producer.
constexpr uint32_t kWarpProducerMinIn = 16;

template <int ES>
__device__ void produce(const KernelArgs& a, const Stage& sm) {
    // The whole warp: lane 0 waits for a free stage and issues the copies;
    // the lanes resolve 32 source addresses at a time (one global load of a
    // buffer id each, all in flight together) and hand them to lane 0.
    const uint32_t lane = threadIdx.x & 31u;
    const uint64_t policy = AR_L2_EVICT_FIRST ? evict_first_policy() : 0;
    uint32_t k = 0;
    bool ok = true;
    for (uint32_t it = blockIdx.x; it < a.n_items; it += gridDim.x, ++k) {
        const WorkItem w = a.items[it];
        const DevProg pg = a.progs[w.prog];
        const uint32_t s = k % a.stages, ph = (k / a.stages) & 1u;
        int free = 0;
        if (lane == 0) free = mbar_wait(sm.empty + 8 * s, ph ^ 1u);
        if (!__shfl_sync(0xFFFFFFFFu, free, 0)) {
            if (lane == 0) atomicOr(a.status, kStatusWaitEmpty);
            ok = false;
            break;
        }
        const uint32_t nb = w.count * ES;
        const uint32_t bar = sm.full + 8 * s;
        if (lane == 0) mbar_expect_tx(bar, nb * pg.n_in);
        const uint32_t dst = sm.tiles + s * sm.stage_bytes;
        for (uint32_t i0 = 0; i0 < pg.n_in; i0 += 32) {
            const char* mine = nullptr;
            if (i0 + lane < pg.n_in) mine = buf_addr(a, a.refs[pg.in_off + i0 + lane]) + w.elem * ES;
            const uint32_t cnt = min(32u, pg.n_in - i0);
            for (uint32_t j = 0; j < cnt; ++j) {
                const char* src = reinterpret_cast<const char*>(
                    __shfl_sync(0xFFFFFFFFu, reinterpret_cast<unsigned long long>(mine), j));
                if (lane == 0) bulk_load(dst + (i0 + j) * a.tile_bytes, src, nb, bar, policy);
            }
        }
    }
    if (!ok && lane == 0) {
        // let the copies already issued land before the CTA can exit
        const uint32_t first = k > static_cast<uint32_t>(a.stages) ? k - a.stages : 0;
        for (uint32_t j = first; j < k; ++j)
            if (!mbar_wait(sm.full + 8 * (j % a.stages), (j / a.stages) & 1u)) atomicOr(a.status, kStatusDrain);
    }
}

// The staged producer for items of few inputs: one thread resolves each
// address and issues its copy.
template <int ES>
__device__ void produce1(const KernelArgs& a, const Stage& sm) {
    const uint64_t policy = AR_L2_EVICT_FIRST ? evict_first_policy() : 0;
    uint32_t k = 0;
    bool ok = true;
    for (uint32_t it = blockIdx.x; it < a.n_items; it += gridDim.x, ++k) {
        const WorkItem w = a.items[it];
        const DevProg pg = a.progs[w.prog];
        const uint32_t s = k % a.stages, ph = (k / a.stages) & 1u;
        if (!mbar_wait(sm.empty + 8 * s, ph ^ 1u)) {
            atomicOr(a.status, kStatusWaitEmpty);
            ok = false;
            break;
        }
        const uint32_t nb = w.count * ES;
        const uint32_t bar = sm.full + 8 * s;
        mbar_expect_tx(bar, nb * pg.n_in);
        const uint32_t dst = sm.tiles + s * sm.stage_bytes;
        for (uint32_t i = 0; i < pg.n_in; ++i) {
            const char* src = buf_addr(a, a.refs[pg.in_off + i]) + w.elem * ES;
            bulk_load(dst + i * a.tile_bytes, src, nb, bar, policy);
        }
    }
    if (!ok) {
        // let the copies already issued land before the CTA can exit
        const uint32_t first = k > static_cast<uint32_t>(a.stages) ? k - a.stages : 0;
        for (uint32_t j = first; j < k; ++j)
            if (!mbar_wait(sm.full + 8 * (j % a.stages), (j / a.stages) & 1u)) atomicOr(a.status, kStatusDrain);
    }
}

template <int DT, int OP, bool RIGHT>
__device__ __forceinline__ void chain_item(const KernelArgs& a, const DevProg& pg, uint32_t st, uint32_t nvec,
                                           int64_t off, int ct) {
    uint4 acc[kVpt];
#pragma unroll
    for (int j = 0; j < kVpt; ++j) {
        const uint32_t v = ct + j * kConsumers;
        if (v < nvec) acc[j] = lds128(st + v * 16);
    }
    for (uint32_t i = 1; i < pg.n_in; ++i) {
        const uint32_t t = st + i * a.tile_bytes;
#pragma unroll
        for (int j = 0; j < kVpt; ++j) {
            const uint32_t v = ct + j * kConsumers;
            if (v < nvec) {
                const uint4 x = lds128(t + v * 16);
                acc[j] = RIGHT ? vop<DT, OP>(x, acc[j]) : vop<DT, OP>(acc[j], x);
            }
        }
    }
    if (pg.flags & PF_AVG) {
#pragma unroll
        for (int j = 0; j < kVpt; ++j) acc[j] = vdiv<DT>(acc[j], static_cast<float>(a.P));
    }
    for (uint32_t o = 0; o < pg.n_out; ++o) {
        char* dst = buf_addr(a, a.refs[pg.out_off + o]) + off;
#pragma unroll
        for (int j = 0; j < kVpt; ++j) {
            const uint32_t v = ct + j * kConsumers;
            if (v < nvec) stg128(dst + v * 16, acc[j]);
        }
    }
}

template <int DT, int OP>
__device__ __forceinline__ void acc_item(const KernelArgs& a, const DevProg& pg, uint32_t st, uint32_t nvec,
                                         int64_t off, int ct) {
    for (uint32_t v = ct; v < nvec; v += kConsumers) {
        const uint4 r = acc_reduce<DT, OP>(pg.n_in, avg_div(a, pg),
                                           [&](uint32_t i) { return lds128(st + i * a.tile_bytes + v * 16); });
        for (uint32_t o = 0; o < pg.n_out; ++o) stg128(buf_addr(a, a.refs[pg.out_off + o]) + off + v * 16, r);
    }
}

template <int DT, int OP>
__device__ __forceinline__ void dag_item(const KernelArgs& a, const DevProg& pg, uint32_t st, uint32_t tmps,
                                         uint32_t nvec, int64_t off, int ct) {
    uint4 acc[kVpt];
    auto ref = [&](uint32_t r) { return (r & REF_TMP) ? tmps + (r & 0x1FFu) * a.tile_bytes : st + r * a.tile_bytes; };
    for (uint32_t q = 0; q < pg.n_ins; ++q) {
        const uint32_t w = a.ins[pg.ins_off + q];
        if ((w >> 30) == INS_OP) {
            const uint32_t ra = w & 0x3FFu, rb = (w >> 10) & 0x3FFu, rd = (w >> 20) & 0x3FFu;
            const uint32_t pa = ref(ra), pb = ref(rb), pd = ref(rd);
#pragma unroll
            for (int j = 0; j < kVpt; ++j) {
                const uint32_t v = ct + j * kConsumers;
                if (v < nvec) {
                    const uint4 x = ra == REF_ACC ? acc[j] : lds128(pa + v * 16);
                    const uint4 y = rb == REF_ACC ? acc[j] : lds128(pb + v * 16);
                    const uint4 r = vop<DT, OP>(x, y);
                    if (rd == REF_ACC)
                        acc[j] = r;
                    else
                        sts128(pd + v * 16, r);
                }
            }
        } else {
            const uint32_t rv = w & 0x3FFu, id = (w >> 10) & 0xFFFFu;
            const uint32_t pv = ref(rv);
            const bool avg = (w >> 30) == INS_STORE_AVG;
            char* dst = buf_addr(a, id) + off;
#pragma unroll
            for (int j = 0; j < kVpt; ++j) {
                const uint32_t v = ct + j * kConsumers;
                if (v < nvec) {
                    const uint4 x = rv == REF_ACC ? acc[j] : lds128(pv + v * 16);
                    stg128(dst + v * 16, avg ? vdiv<DT>(x, static_cast<float>(a.P)) : x);
                }
            }
        }
    }
}

// Dag: how the launch evaluates DAG programs, called as
// dag(pg, prog_index, stage_tiles, nvec, byte_offset, consumer_thread).
// Forced inline like everything between the kernel and the programs: a
// called function reaches the kernel parameters through a pointer, and then
// every store may overwrite them, so buffer addresses are reloaded from
// memory after each store.
template <int DT, int OP, class Dag>
__device__ __forceinline__ void consume(const KernelArgs& a, const Stage& sm, int ct, Dag dag) {
    constexpr int ES = DT == AR_BFLOAT16 ? 2 : 4;
    const int lane = ct & 31;
    uint32_t k = 0;
    for (uint32_t it = blockIdx.x; it < a.n_items; it += gridDim.x, ++k) {
        const WorkItem w = a.items[it];
        const DevProg pg = a.progs[w.prog];
        const uint32_t s = k % a.stages, ph = (k / a.stages) & 1u;
        if (!mbar_wait(sm.full + 8 * s, ph)) {
            atomicOr(a.status, kStatusWaitFull);
            return;
        }
        const uint32_t st = sm.tiles + s * sm.stage_bytes;
        const uint32_t nvec = (w.count * ES) >> 4;
        const int64_t off = w.elem * ES;
        if (pg.kind == PK_CHAIN_R)
            chain_item<DT, OP, true>(a, pg, st, nvec, off, ct);
        else if (pg.kind == PK_CHAIN_L)
            chain_item<DT, OP, false>(a, pg, st, nvec, off, ct);
        else if (pg.kind == PK_ACC)
            acc_item<DT, OP>(a, pg, st, nvec, off, ct);
        else if (pg.kind == PK_TREE)
            atomicOr(a.status, kStatusBadProgram);  // trees run on the rank-streaming kernel
        else
            dag(pg, w.prog, st, nvec, off, ct);
        __syncwarp();
        if (lane == 0) mbar_arrive(sm.empty + 8 * s);
    }
}

// Binds the stage layout to a launch's DAG evaluator (a functor, not a
// lambda, so that its call can be forced inline).
template <class Dag>
struct StagedDag {
    const Stage& sm;
    const Dag& dag;
    __device__ __forceinline__ void operator()(const DevProg& pg, uint32_t prog, uint32_t st, uint32_t nvec,
                                               int64_t off, int ct) const {
        dag(sm, pg, prog, st, nvec, off, ct);
    }
};

// The staged kernel: barrier setup, one producer thread, eight consumer
// warps.  smem is the dynamic shared memory; dag evaluates DAG programs.
template <int DT, int OP, class Dag>
__device__ __forceinline__ void staged_body(const KernelArgs& a, uint8_t* smem, Dag dag) {
    constexpr int ES = DT == AR_BFLOAT16 ? 2 : 4;
    Stage sm;
    sm.full = smem_addr(smem);
    sm.empty = sm.full + 8 * a.stages;
    sm.tiles = sm.full + kBarrierBytes;
    sm.stage_bytes = static_cast<uint32_t>(a.tile_bytes) * a.max_in;
    sm.tmps = sm.tiles + a.stages * sm.stage_bytes;
    if (threadIdx.x == 0) {
        for (int s = 0; s < a.stages; ++s) {
            mbar_init(sm.full + 8 * s, 1);
            mbar_init(sm.empty + 8 * s, kConsumerWarps);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    griddep_wait();
    griddep_launch_dependents();
    if (threadIdx.x < 32) {
        // many inputs per item: the whole warp resolves the addresses
        // (measured +15-20 points of the copy peak at P = 31 ... 64); few:
        // one thread (the warp's shuffles cost 30-40 points at P = 7 ... 16)
        if (a.max_in > kWarpProducerMinIn)
            produce<ES>(a, sm);
        else if (threadIdx.x == 0)
            produce1<ES>(a, sm);
        return;
    }
    consume<DT, OP>(a, sm, threadIdx.x - 32, StagedDag<Dag>{sm, dag});
}

}  // namespace
}  // namespace ar
