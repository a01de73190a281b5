// CUDA kernels of the allreduce engine (sm_103a).
//
// staged_kernel: persistent, one CTA per SM, warp-specialised.  Lane 0 of
// warp 0 is the producer: for every work item it waits for a free pipeline
// stage and issues one cp.async.bulk (TMA bulk copy) per input buffer of the
// item's program into that stage, completing on the stage's mbarrier.  Eight
// consumer warps wait for the stage, evaluate the tile program from shared
// memory (chains and DAG instructions on 16-byte vectors, one accumulator
// register per vector) and store the results to global memory with 128-bit
// streaming stores, then release the stage.  Every wait is bounded: after two
// seconds the waiter sets a bit in the plan's status word and the CTA winds
// down (the producer first waits, again bounded, for its copies in flight).
//
// elementwise_kernel: one CTA per work item, one element per thread; used for
// the unaligned heads / tails of ranges and for buffers that are not 16-byte
// aligned.  Same programs, same arithmetic, same accumulation order.
//
// Element arithmetic (sum / prod / max / min over int32, fp32, bf16): int32
// wraps, fp32 uses IEEE round-to-nearest-even adds and multiplies without
// contraction or flushing, bf16 widens to fp32, applies the fp32 op and
// rounds back to bf16 to nearest even after every op; max is a > b ? a : b
// and min a < b ? a : b.
#include <cstdint>

#include "kernels.hpp"

namespace ar {
namespace {

constexpr uint64_t kWaitNs = 2000000000ull;  // bounded waits give up after 2 s
constexpr int kVpt = 8;                      // 16-byte vectors per consumer thread per item
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

// a (+) b on one 32-bit word: one int32 / fp32 element or two bf16 elements
template <int DT, int OP>
__device__ __forceinline__ uint32_t wop(uint32_t a, uint32_t b) {
    if (DT == AR_INT32) return static_cast<uint32_t>(iop<OP>(static_cast<int32_t>(a), static_cast<int32_t>(b)));
    if (DT == AR_FLOAT32) return __float_as_uint(fop<OP>(__uint_as_float(a), __uint_as_float(b)));
    const float al = bf_lo(a), ah = bf_hi(a), bl = bf_lo(b), bh = bf_hi(b);
    if (OP == AR_MAX || OP == AR_MIN) {
        const bool pl = OP == AR_MAX ? al > bl : al < bl;
        const bool ph = OP == AR_MAX ? ah > bh : ah < bh;
        return ((pl ? a : b) & 0xFFFFu) | ((ph ? a : b) & 0xFFFF0000u);
    }
    return pack_bf16x2(fop<OP>(al, bl), fop<OP>(ah, bh));
}

template <int DT, int OP>
__device__ __forceinline__ uint4 vop(uint4 a, uint4 b) {
    return make_uint4(wop<DT, OP>(a.x, b.x), wop<DT, OP>(a.y, b.y), wop<DT, OP>(a.z, b.z),
                      wop<DT, OP>(a.w, b.w));
}

// Accumulator of the FP32ACC order: int32 stays int32 (exact in any order),
// fp32 and bf16 accumulate in fp32 and round once.
template <int DT>
struct Acc {
    static constexpr int W = DT == AR_BFLOAT16 ? 8 : 4;
    float f[W];
    int32_t i[4];
};

template <int DT, int OP>
__device__ __forceinline__ void acc_identity(Acc<DT>& x) {
    if (DT == AR_INT32) {
        const int32_t id = OP == AR_SUM ? 0 : OP == AR_PROD ? 1 : OP == AR_MAX ? INT32_MIN : INT32_MAX;
#pragma unroll
        for (int q = 0; q < 4; ++q) x.i[q] = id;
    } else {
        const float id = OP == AR_SUM ? -0.0f : OP == AR_PROD ? 1.0f : OP == AR_MAX ? -INFINITY : INFINITY;
#pragma unroll
        for (int q = 0; q < Acc<DT>::W; ++q) x.f[q] = id;
    }
}

template <int DT>
__device__ __forceinline__ void acc_widen(Acc<DT>& x, uint4 v) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    if (DT == AR_INT32) {
#pragma unroll
        for (int q = 0; q < 4; ++q) x.i[q] = static_cast<int32_t>(w[q]);
    } else if (DT == AR_FLOAT32) {
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
    if (DT == AR_INT32) {
#pragma unroll
        for (int q = 0; q < 4; ++q) x.i[q] = iop<OP>(x.i[q], y.i[q]);
    } else {
#pragma unroll
        for (int q = 0; q < Acc<DT>::W; ++q) x.f[q] = fop<OP>(x.f[q], y.f[q]);
    }
}

template <int DT>
__device__ __forceinline__ uint4 acc_narrow(const Acc<DT>& x) {
    if (DT == AR_INT32)
        return make_uint4(static_cast<uint32_t>(x.i[0]), static_cast<uint32_t>(x.i[1]),
                          static_cast<uint32_t>(x.i[2]), static_cast<uint32_t>(x.i[3]));
    if (DT == AR_FLOAT32)
        return make_uint4(__float_as_uint(x.f[0]), __float_as_uint(x.f[1]), __float_as_uint(x.f[2]),
                          __float_as_uint(x.f[3]));
    return make_uint4(pack_bf16x2(x.f[0], x.f[1]), pack_bf16x2(x.f[2], x.f[3]), pack_bf16x2(x.f[4], x.f[5]),
                      pack_bf16x2(x.f[6], x.f[7]));
}

// FP32ACC order over n inputs: blocks of 8 consecutive inputs reduced as a
// balanced pairwise tree (missing inputs are the op's identity), block
// results folded left to right.  load(i) yields input i as a 16-byte vector.
template <int DT, int OP, class Load>
__device__ __forceinline__ uint4 acc_reduce(uint32_t n, Load load) {
    Acc<DT> acc;
    for (uint32_t g = 0; g < n; g += 8) {
        Acc<DT> s[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            if (g + q < n)
                acc_widen<DT>(s[q], load(g + q));
            else
                acc_identity<DT, OP>(s[q]);
        }
        acc_combine<DT, OP>(s[0], s[1]);
        acc_combine<DT, OP>(s[2], s[3]);
        acc_combine<DT, OP>(s[4], s[5]);
        acc_combine<DT, OP>(s[6], s[7]);
        acc_combine<DT, OP>(s[0], s[2]);
        acc_combine<DT, OP>(s[4], s[6]);
        acc_combine<DT, OP>(s[0], s[4]);
        if (g == 0)
            acc = s[0];
        else
            acc_combine<DT, OP>(acc, s[0]);
    }
    return acc_narrow<DT>(acc);
}

// ------------------------------------------------------------- memory access

__device__ __forceinline__ char* buf_addr(const KernelArgs& a, uint32_t id) {
    const uint32_t slot = id >> 6, rank = id & 63u;
    if (slot == 0) return static_cast<char*>(a.bufs[rank]);
    return a.scratch + (static_cast<uint64_t>(slot - 1) * a.P + rank) * a.slot_stride;
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

__device__ __forceinline__ void sts128(uint32_t addr, uint4 v) {
    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z),
                 "r"(v.w)
                 : "memory");
}

__device__ __forceinline__ void stg128(char* p, uint4 v) {
    asm volatile("st.global.cs.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
                 "r"(v.w)
                 : "memory");
}

__device__ __forceinline__ uint64_t globaltimer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
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

// Waits for the phase of the given parity; false after kWaitNs.
__device__ __noinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer();
    for (;;) {
        for (int i = 0; i < 32; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (globaltimer() - t0 > kWaitNs) return false;
    }
}

__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

// ------------------------------------------------------------ staged kernel

struct Stage {
    uint32_t full, empty;  // mbarrier arrays (shared addresses)
    uint32_t tiles;        // stage 0 tiles
    uint32_t tmps;         // temporaries
    uint32_t stage_bytes;
};

template <int ES>
__device__ void produce(const KernelArgs& a, const Stage& sm) {
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
            bulk_load(dst + i * a.tile_bytes, src, nb, bar);
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
        const uint4 r = acc_reduce<DT, OP>(pg.n_in, [&](uint32_t i) { return lds128(st + i * a.tile_bytes + v * 16); });
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
            char* dst = buf_addr(a, id) + off;
#pragma unroll
            for (int j = 0; j < kVpt; ++j) {
                const uint32_t v = ct + j * kConsumers;
                if (v < nvec) stg128(dst + v * 16, rv == REF_ACC ? acc[j] : lds128(pv + v * 16));
            }
        }
    }
}

template <int DT, int OP>
__device__ void consume(const KernelArgs& a, const Stage& sm, int ct) {
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
        else
            dag_item<DT, OP>(a, pg, st, sm.tmps, nvec, off, ct);
        __syncwarp();
        if (lane == 0) mbar_arrive(sm.empty + 8 * s);
    }
}

template <int DT, int OP>
__global__ void __launch_bounds__(kStagedThreads, 1) staged_kernel(const __grid_constant__ KernelArgs a) {
    extern __shared__ __align__(128) uint8_t smem[];
    constexpr int ES = DT == AR_BFLOAT16 ? 2 : 4;
    Stage sm;
    sm.full = smem_addr(smem);
    sm.empty = sm.full + 8 * a.stages;
    sm.tiles = sm.full + 128;
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
    if (threadIdx.x < 32) {
        if (threadIdx.x == 0) produce<ES>(a, sm);
        return;
    }
    consume<DT, OP>(a, sm, threadIdx.x - 32);
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

template <int DT, int OP>
__global__ void __launch_bounds__(kElemThreads) elementwise_kernel(const __grid_constant__ KernelArgs a) {
    extern __shared__ uint32_t vals[];  // [(max_in + max_tmp) rows][kElemThreads]
    constexpr int ES = DT == AR_BFLOAT16 ? 2 : 4;
    const WorkItem w = a.items[blockIdx.x];
    const DevProg pg = a.progs[w.prog];
    const int t = threadIdx.x;
    auto row = [&](uint32_t r) -> uint32_t& {
        return (r & REF_TMP) ? vals[(a.max_in + (r & 0x1FFu)) * kElemThreads + t] : vals[r * kElemThreads + t];
    };
    for (uint32_t e = t; e < w.count; e += kElemThreads) {
        const int64_t off = (w.elem + e) * ES;
        for (uint32_t i = 0; i < pg.n_in; ++i)
            vals[i * kElemThreads + t] = ld_elem<DT>(buf_addr(a, a.refs[pg.in_off + i]) + off);
        if (pg.kind == PK_CHAIN_R || pg.kind == PK_CHAIN_L) {
            uint32_t acc = vals[t];
            for (uint32_t i = 1; i < pg.n_in; ++i) {
                const uint32_t x = vals[i * kElemThreads + t];
                acc = pg.kind == PK_CHAIN_R ? eop<DT, OP>(x, acc) : eop<DT, OP>(acc, x);
            }
            for (uint32_t o = 0; o < pg.n_out; ++o) st_elem<DT>(buf_addr(a, a.refs[pg.out_off + o]) + off, acc);
        } else if (pg.kind == PK_ACC) {
            // same order as the staged kernel: the element sits in lane 0 of a
            // vector whose other lanes hold the op's identity-free zeros; only
            // lane 0 of the result is kept
            const uint4 r = acc_reduce<DT, OP>(pg.n_in, [&](uint32_t i) {
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
                    st_elem<DT>(buf_addr(a, id) + off, rv == REF_ACC ? acc : row(rv));
                }
            }
        }
    }
}

// ----------------------------------------------------------------- dispatch

using KernelFn = void (*)(KernelArgs);

template <int DT, int OP>
struct Table {
    static constexpr KernelFn staged = staged_kernel<DT, OP>;
    static constexpr KernelFn elem = elementwise_kernel<DT, OP>;
};

template <int DT>
KernelFn pick(int op, bool staged) {
    switch (op) {
        case AR_SUM: return staged ? Table<DT, AR_SUM>::staged : Table<DT, AR_SUM>::elem;
        case AR_PROD: return staged ? Table<DT, AR_PROD>::staged : Table<DT, AR_PROD>::elem;
        case AR_MAX: return staged ? Table<DT, AR_MAX>::staged : Table<DT, AR_MAX>::elem;
        default: return staged ? Table<DT, AR_MIN>::staged : Table<DT, AR_MIN>::elem;
    }
}

KernelFn kernel_for(int dtype, int op, bool staged) {
    switch (dtype) {
        case AR_INT32: return pick<AR_INT32>(op, staged);
        case AR_FLOAT32: return pick<AR_FLOAT32>(op, staged);
        default: return pick<AR_BFLOAT16>(op, staged);
    }
}

}  // namespace

cudaError_t prepare_kernels(int dtype, int op) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    int optin = 0;
    e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (e != cudaSuccess) return e;
    for (bool staged : {true, false}) {
        e = cudaFuncSetAttribute(reinterpret_cast<const void*>(kernel_for(dtype, op, staged)),
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, optin);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

cudaError_t launch_staged(int dtype, int op, const KernelArgs& a, int grid, int smem, cudaStream_t st) {
    KernelFn f = kernel_for(dtype, op, true);
    f<<<grid, kStagedThreads, smem, st>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_elementwise(int dtype, int op, const KernelArgs& a, int smem, cudaStream_t st) {
    KernelFn f = kernel_for(dtype, op, false);
    f<<<a.n_items, kElemThreads, smem, st>>>(a);
    return cudaGetLastError();
}

}  // namespace ar
