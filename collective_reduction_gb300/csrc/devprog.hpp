// Tile programs: the device-side form of a compiled schedule.
//
// A work item is an element range of every rank buffer with one program.
// The program lists the buffers to load (inputs, in order), then either
//   CHAIN_R  acc = in[0]; acc = in[i] (+) acc for i = 1..n_in-1   (ring order)
//   CHAIN_L  acc = in[0]; acc = acc (+) in[i]
//   ACC      fp32 accumulation of all inputs in the kernel's fixed order
//   TREE     one tree evaluated in post-order on a stack: push in[i], then
//            c_i times replace the two top entries a, b by a (+) b, where c_i
//            is bits 4(i mod 8)..+3 of ins[i / 8]
// followed by storing acc (the tree: the last stack entry) to every output
// buffer, or
//   DAG      a straight-line list of instructions over inputs, temporaries
//            and one accumulator register: OP d = a (+) b, STORE buf <- v.
// All inputs of an item are loaded before any output is stored, so a
// program may overwrite buffers it reads (the step form relies on this).
#pragma once

#if !defined(__CUDACC_RTC__)
#include <cstdint>
#endif

#if defined(__CUDACC__)
#define AR_HD __host__ __device__
#else
#define AR_HD
#endif

namespace ar {

enum ProgKind : uint8_t { PK_CHAIN_R = 0, PK_CHAIN_L = 1, PK_DAG = 2, PK_ACC = 3, PK_TREE = 4 };
// DevProg::flags: the outputs are every rank's own buffer in rank order, so a
// kernel can take output o's address straight from the rank-pointer array
constexpr uint8_t PF_OUT_ALL = 1;
// DevProg::flags: the program's result is a complete AR_AVG sum, divided by P
// before it is stored
constexpr uint8_t PF_AVG = 2;

// value references inside DAG instructions (10 bits)
constexpr uint32_t REF_TMP = 0x200;  // bit 9 set: temporary index in bits 0..8
constexpr uint32_t REF_ACC = 0x3FF;  // the accumulator register
constexpr uint32_t MAX_IN = 256;     // inputs per program
constexpr uint32_t MAX_TMP = 511;    // temporaries per program
constexpr int kBarrierBytes = 512;   // mbarrier area at the start of a kernel's shared memory

// Kernel geometry the lowering must agree with: consumer warps per CTA of the
// staged / rank-streaming kernels, 16-byte vectors each consumer thread takes
// per item tile (staged: up to kStagedVpt) or per rank tile (streaming).
constexpr int kConsumerWarps = 8;
constexpr int kElemBlock = 64;       // element-wise kernel: threads = elements per block
constexpr int kStagedVpt = 4;
constexpr int kStreamVpt = 8;        // rank-streaming kernel, chains and fp32 / int32 accumulation
constexpr int kStreamVptTree = 6;    // rank-streaming kernel: trees deeper than the wide tiles allow, bf16 fp32 accumulation
constexpr int kMaxStagedTile = 32 * kConsumerWarps * 16 * kStagedVpt;          // 16 KB
// chain word kernel: threads per CTA (one 32-bit word each per item pass),
// most inputs / outputs of a program it runs
constexpr int kChainWordThreads = 128;
constexpr int kCopyThreads = 256;  // the copy kernel (one input, many outputs)
constexpr int kFewMaxIn = 16;        // the few-input kernel: most inputs of a program
constexpr int kFewTreeMaxIn = 8;     // ... of a single tree
// ... and the stack entries below the top of a tree its instantiation for
// trees of up to m leaves holds
AR_HD constexpr int few_tree_stack(int m) { return m <= 4 ? 2 : 4; }
constexpr int kChainWordMaxIn = 64;
constexpr int kStreamTileBytes = 32 * kConsumerWarps * 16 * kStreamVpt;        // 32 KB
constexpr int kStreamTileTree = 32 * kConsumerWarps * 16 * kStreamVptTree;     // 24 KB
// TREE programs: leaves in post-order, and after each leaf the number of
// combines that follow it (4 bits per leaf, 8 leaves per instruction word).
// Evaluated with the deeper child first, a tree of at most 64 leaves needs a
// stack of at most 7 entries; DevProg::n_tmp holds the program's depth - 1.
constexpr int kTreeDepth = 7;
constexpr int kTreeMaxLeaves = 64;
constexpr int kTreeCountWords = kTreeMaxLeaves / 8;

// instruction word: bits 30..31 kind
//   OP:    a = bits 0..9, b = bits 10..19, d = bits 20..29
//   STORE: v = bits 0..9, buffer id = bits 10..25
//   STORE_AVG: as STORE, the value divided by P first (AR_AVG results)
constexpr uint32_t INS_OP = 0u;
constexpr uint32_t INS_STORE = 1u;
constexpr uint32_t INS_STORE_AVG = 2u;

AR_HD inline uint32_t ins_op(uint32_t a, uint32_t b, uint32_t d) {
    return (INS_OP << 30) | a | (b << 10) | (d << 20);
}
AR_HD inline uint32_t ins_store(uint32_t v, uint32_t buf, bool avg = false) {
    return ((avg ? INS_STORE_AVG : INS_STORE) << 30) | v | (buf << 10);
}

// Buffer id: (slot << 6) | rank.  Slot 0 is the rank's own buffer; slot s >= 1
// lives in the plan's scratch at ((s - 1) * P + rank) * slot_stride bytes.
AR_HD inline uint32_t buf_id(int slot, int rank) {
    return (static_cast<uint32_t>(slot) << 6) | static_cast<uint32_t>(rank);
}

struct DevProg {
    uint8_t kind;
    uint8_t flags;
    uint16_t n_in;
    uint16_t n_tmp;
    uint16_t n_out;     // CHAIN / ACC: number of output buffers
    uint32_t n_ins;     // DAG: number of instruction words
    uint32_t in_off;    // refs[in_off ..): input buffer ids
    uint32_t out_off;   // refs[out_off ..): output buffer ids (CHAIN / ACC)
    uint32_t ins_off;   // ins[ins_off ..): instruction words (DAG)
};

struct WorkItem {
    int64_t elem;       // first element of the range
    uint32_t count;     // elements in the range
    uint32_t prog;      // program index
};

}  // namespace ar
