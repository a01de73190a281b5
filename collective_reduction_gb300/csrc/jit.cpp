// Run-time compiled DAG kernels: source generation, NVRTC compilation and
// loading (see jit.hpp).
#include "jit.hpp"

#include <cuda_runtime.h>
#include <dlfcn.h>

#include <algorithm>
#include <cstdio>
#include <functional>
#include <map>
#include <mutex>
#include <set>
#include <sstream>
#include <stdexcept>
#include <string>
#include <vector>

#include "kargs.hpp"

namespace ar {
namespace {

// The headers the generated source includes, embedded at build time.
#include "jit_headers.inc"

// DAG programs used by bulk items of staged (non-streaming) launches.
std::set<uint32_t> staged_dag_programs(const Lowered& L) {
    std::set<uint32_t> ids;
    for (const LaunchSet& s : L.sets) {
        if (s.stream || s.small || s.words) continue;
        for (const WorkItem& w : s.bulk)
            if (L.progs[w.prog].kind == PK_DAG) ids.insert(w.prog);
    }
    return ids;
}

// Straight-line code of one DAG program over this thread's vectors of an
// item: leaves are loaded from their stage tiles at first use, every result
// is a new register value, stores go to addresses computed once per item.
void emit_program(std::ostringstream& o, const Lowered& L, uint32_t id, int P) {
    const DevProg& d = L.progs[id];
    std::map<uint32_t, int> outs;  // buffer id -> pointer index
    for (uint32_t q = 0; q < d.n_ins; ++q) {
        const uint32_t w = L.ins[d.ins_off + q];
        if ((w >> 30) != INS_OP) outs.emplace((w >> 10) & 0xFFFFu, static_cast<int>(outs.size()));
    }
    o << "__device__ __forceinline__ void dag_" << id
      << "(const KernelArgs& a, uint32_t st, uint32_t nvec, int64_t off, int ct) {\n";
    for (const auto& kv : outs) o << "    char* const o" << kv.second << " = buf_addr(a, " << kv.first << "u) + off;\n";
    o << "#pragma unroll 1\n"
         "    for (int j = 0; j < kVpt; ++j) {\n"
         "        const uint32_t v = ct + j * kConsumers;\n"
         "        if (v >= nvec) break;\n"
         "        const uint32_t s = st + v * 16u;\n";
    std::vector<char> loaded(d.n_in, 0);
    std::map<uint32_t, std::string> tmp;  // temporary slot -> current value
    std::string acc;
    int fresh = 0;
    auto value = [&](uint32_t r) -> std::string {
        if (r == REF_ACC) return acc;
        if (r & REF_TMP) return tmp.at(r & 0x1FFu);
        if (r >= d.n_in) throw std::logic_error("dag program reads a missing input");
        if (!loaded[r]) {
            o << "        const uint4 x" << r << " = lds128(s + " << static_cast<uint64_t>(r) * L.tile_bytes << "u);\n";
            loaded[r] = 1;
        }
        return "x" + std::to_string(r);
    };
    for (uint32_t q = 0; q < d.n_ins; ++q) {
        const uint32_t w = L.ins[d.ins_off + q];
        if ((w >> 30) == INS_OP) {
            const std::string x = value(w & 0x3FFu), y = value((w >> 10) & 0x3FFu);
            const std::string t = "t" + std::to_string(fresh++);
            o << "        const uint4 " << t << " = vop<DT, OP>(" << x << ", " << y << ");\n";
            const uint32_t rd = (w >> 20) & 0x3FFu;
            if (rd == REF_ACC)
                acc = t;
            else
                tmp[rd & 0x1FFu] = t;
        } else {
            const std::string x = value(w & 0x3FFu);
            const int ptr = outs.at((w >> 10) & 0xFFFFu);
            if ((w >> 30) == INS_STORE_AVG)
                o << "        stg128(o" << ptr << " + v * 16u, vdiv<DT>(" << x << ", " << P << ".0f));\n";
            else
                o << "        stg128(o" << ptr << " + v * 16u, " << x << ");\n";
        }
    }
    o << "    }\n}\n\n";
}

// Programs used by bulk items of word-kernel launches.
std::set<uint32_t> word_programs(const Lowered& L) {
    std::set<uint32_t> ids;
    for (const LaunchSet& s : L.sets) {
        if (!s.words) continue;
        for (const WorkItem& w : s.bulk) ids.insert(w.prog);
    }
    return ids;
}

// Address expression of buffer id at byte position `pos` (P ranks).
std::string word_addr(uint32_t id, int P, bool out, const char* pos) {
    const uint32_t slot = id >> 6, rank = id & 63u;
    std::ostringstream o;
    if (slot == 0)
        o << "static_cast<" << (out ? "char*" : "const char*") << ">(a.bufs[" << rank << "])";
    else
        o << "(a.scratch + " << static_cast<uint64_t>(slot - 1) * P + rank << "ull * a.slot_stride)";
    o << " + " << pos;
    return o.str();
}

// One combine of a DAG program in SSA form: operand values a and b (values
// below n_in are the inputs, n_in + k is combine k) and its depth above the
// inputs.
struct DagOp {
    int a, b, level;
};

// The order a word consumer evaluates the combines in: each combine after
// the combines it reads, by depth above the inputs, in list order within a
// depth.  (Choosing among the ready combines the one that ends the most
// values and starts the fewest cut the peak of live values from 143 to 128
// at P = 63 and from 97 to 66 at P = 64 RD, but measured -5 ... +4 points
// of the copy peak, plan by plan: the compiler schedules the loads anyway.)
std::vector<int> dag_order(const std::vector<DagOp>& ops) {
    std::vector<int> order(ops.size());
    for (size_t k = 0; k < ops.size(); ++k) order[k] = static_cast<int>(k);
    std::stable_sort(order.begin(), order.end(), [&](int x, int y) { return ops[x].level < ops[y].level; });
    return order;
}

// The combines and stores of one program over 32-bit words, at byte
// position `pos` of every buffer: input(i) names input word i (emitting its
// load when the variant loads at first use).  Chains fold in their order; a
// DAG program runs in SSA form level by level (each combine after the
// combines it reads, by its depth above the inputs: the same combines of the
// same values as the instruction list, with fewer values live at once).
void emit_word_body(std::ostringstream& o, const Lowered& L, const DevProg& d, int P,
                    const std::function<std::string(uint32_t)>& input) {
    auto store = [&](uint32_t buf, const std::string& v, bool avg) {
        o << "        stg32(" << word_addr(buf, P, true, "pos") << ", "
          << (avg ? "wdiv<DT>(" + v + ", " + std::to_string(P) + ".0f)" : v) << ");\n";
    };
    if (d.kind == PK_CHAIN_R || d.kind == PK_CHAIN_L) {
        std::string acc = input(0);
        for (uint32_t i = 1; i < d.n_in; ++i) {
            const std::string x = input(i);
            const std::string t = "c" + std::to_string(i);
            o << "        const uint32_t " << t << " = wop<DT, OP>(" << (d.kind == PK_CHAIN_R ? x + ", " + acc : acc + ", " + x)
              << ");\n";
            acc = t;
        }
        const bool avg = (d.flags & PF_AVG) != 0;
        for (uint32_t q = 0; q < d.n_out; ++q)
            store((d.flags & PF_OUT_ALL) ? buf_id(0, static_cast<int>(q)) : L.refs[d.out_off + q], acc, avg);
        return;
    }
    if (d.kind != PK_DAG) throw std::logic_error("word kernel: a program kind it does not run");
    std::vector<DagOp> ops;  // value n_in + k is ops[k]
    std::vector<std::pair<uint32_t, std::pair<int, bool>>> stores;  // (buffer, (value, avg))
    std::map<uint32_t, int> tmp;
    int acc = -1;
    auto value = [&](uint32_t r) -> int {
        if (r == REF_ACC) return acc;
        if (r & REF_TMP) return tmp.at(r & 0x1FFu);
        if (r >= d.n_in) throw std::logic_error("dag program reads a missing input");
        return static_cast<int>(r);
    };
    auto level = [&](int v) { return v < static_cast<int>(d.n_in) ? 0 : ops[v - d.n_in].level; };
    for (uint32_t q = 0; q < d.n_ins; ++q) {
        const uint32_t w = L.ins[d.ins_off + q];
        if ((w >> 30) == INS_OP) {
            const int x = value(w & 0x3FFu), y = value((w >> 10) & 0x3FFu);
            if (x < 0 || y < 0) throw std::logic_error("dag program reads an unset accumulator");
            ops.push_back({x, y, std::max(level(x), level(y)) + 1});
            const int v = static_cast<int>(d.n_in + ops.size() - 1);
            const uint32_t rd = (w >> 20) & 0x3FFu;
            if (rd == REF_ACC)
                acc = v;
            else
                tmp[rd & 0x1FFu] = v;
        } else {
            const int v = value(w & 0x3FFu);
            if (v < 0) throw std::logic_error("dag program stores an unset accumulator");
            stores.push_back({(w >> 10) & 0xFFFFu, {v, (w >> 30) == INS_STORE_AVG}});
        }
    }
    const std::vector<int> order = dag_order(ops);
    auto name = [&](int v) -> std::string {
        return v < static_cast<int>(d.n_in) ? input(static_cast<uint32_t>(v)) : "t" + std::to_string(v - d.n_in);
    };
    std::map<int, std::vector<size_t>> stores_of;
    for (size_t k = 0; k < stores.size(); ++k) stores_of[stores[k].second.first].push_back(k);
    auto emit_stores = [&](int v) {
        auto it = stores_of.find(v);
        if (it == stores_of.end()) return;
        const std::string x = name(v);
        for (size_t k : it->second) store(stores[k].first, x, stores[k].second.second);
    };
    for (uint32_t i = 0; i < d.n_in; ++i) emit_stores(static_cast<int>(i));
    for (int k : order) {
        const std::string x = name(ops[k].a), y = name(ops[k].b);
        o << "        const uint32_t t" << k << " = wop<DT, OP>(" << x << ", " << y << ");\n";
        emit_stores(static_cast<int>(d.n_in) + k);
    }
}

// Address expression of input word i of program d at byte position q.
std::string word_src(const Lowered& L, const DevProg& d, uint32_t i, int P, const char* q) {
    return word_addr(L.refs[d.in_off + i], P, false, q);
}

// One program over 32-bit words, each thread taking word positions t,
// t + kWordThreads, ... of the item.  Direct (stages = 0): every input word of
// a position is loaded into registers before any store (a program may store
// to a buffer it reads).  Prefetching (stages = S >= 2): the thread copies the
// input words of the position S - 1 ahead with 4-byte asynchronous copies
// (no registers held while they are in flight) into its own slots of stage
// (position mod S) — [stage][input][thread], so a warp's copies and reads are
// 128 contiguous bytes — waits for the current position's group and reads each
// word at its first use; the prefetched positions are never the ones being
// stored, and a stage is refilled only after its words were read.
void emit_word_program(std::ostringstream& o, const Lowered& L, uint32_t id, int P, int threads, int S) {
    const DevProg& d = L.progs[id];
    o << "__device__ __forceinline__ void wp_" << id
      << "(const KernelArgs& a, int64_t off, uint32_t nw, uint32_t sbase) {\n";
    if (S == 0) {
        o << "#pragma unroll 1\n"
             "    for (uint32_t t = threadIdx.x; t < nw; t += "
          << threads << "u) {\n        const int64_t pos = off + 4 * static_cast<int64_t>(t);\n";
        for (uint32_t i = 0; i < d.n_in; ++i)
            o << "        const uint32_t x" << i << " = ldg32(" << word_src(L, d, i, P, "pos") << ");\n";
        emit_word_body(o, L, d, P, [](uint32_t i) { return "x" + std::to_string(i); });
        o << "    }\n}\n\n";
        return;
    }
    const uint64_t islot = 4ull * threads;  // bytes between inputs in a stage
    const uint64_t sstage = islot * d.n_in;  // bytes of one stage of this program
    auto prefetch = [&](const char* tvar, const char* kvar, const char* indent) {
        o << indent << "if (" << tvar << " < nw) {\n";
        o << indent << "    const int64_t q = off + 4 * static_cast<int64_t>(" << tvar << ");\n";
        o << indent << "    const uint32_t d = sb + " << kvar << " * " << sstage << "u;\n";
        for (uint32_t i = 0; i < d.n_in; ++i)
            o << indent << "    cp_async4(d + " << i * islot << "u, " << word_src(L, d, i, P, "q") << ");\n";
        o << indent << "}\n" << indent << "cp_async_commit();\n";
    };
    o << "    const uint32_t sb = sbase + 4u * threadIdx.x;\n";
    for (int k = 0; k + 1 < S; ++k) {
        o << "    {\n        const uint32_t tp = threadIdx.x + " << k * threads << "u;\n        const uint32_t kp = " << k
          << "u;\n";
        prefetch("tp", "kp", "        ");
        o << "    }\n";
    }
    o << "    uint32_t k = 0;\n"
         "#pragma unroll 1\n"
         "    for (uint32_t t = threadIdx.x; t < nw; t += "
      << threads << "u, k = (k + 1 == " << S << "u ? 0u : k + 1)) {\n";
    o << "        {\n            const uint32_t tn = t + " << (S - 1) * threads << "u;\n"
      << "            const uint32_t kn = (k + " << (S - 1) << "u) % " << S << "u;\n";
    prefetch("tn", "kn", "            ");
    o << "        }\n        cp_async_wait<" << S - 1 << ">();\n        const uint32_t s = sb + k * " << sstage
      << "u;\n        const int64_t pos = off + 4 * static_cast<int64_t>(t);\n";
    std::vector<char> loaded(d.n_in, 0);
    emit_word_body(o, L, d, P, [&](uint32_t i) -> std::string {
        if (i >= d.n_in) throw std::logic_error("word program reads a missing input");
        if (!loaded[i]) {
            o << "        const uint32_t x" << i << " = lds32(s + " << i * islot << "u);\n";
            loaded[i] = 1;
        }
        return "x" + std::to_string(i);
    });
    o << "    }\n    cp_async_wait<0>();\n}\n\n";
}

// A DAG program of the staged kernel over 32-bit words (programs of many
// inputs, whose 16-byte vectors would not all fit in registers): each
// consumer thread takes words ct, ct + kConsumers, ... of the item's tiles,
// loads an input word from its stage tile at first use, and evaluates the
// instruction list in SSA form level by level (an op after the ops it
// reads, in order of its depth above the inputs: the same combines of the
// same values as the list's order, with fewer values live at once), storing
// each result word straight to its output.
void emit_program_words(std::ostringstream& o, const Lowered& L, uint32_t id, int P) {
    const DevProg& d = L.progs[id];
    std::vector<DagOp> ops;  // value n_in + k is ops[k]
    std::vector<std::pair<uint32_t, std::pair<int, bool>>> stores;  // (buffer, (value, avg))
    std::map<uint32_t, int> tmp;
    int acc = -1;
    auto value = [&](uint32_t r) -> int {
        if (r == REF_ACC) return acc;
        if (r & REF_TMP) return tmp.at(r & 0x1FFu);
        if (r >= d.n_in) throw std::logic_error("dag program reads a missing input");
        return static_cast<int>(r);
    };
    auto level = [&](int v) { return v < static_cast<int>(d.n_in) ? 0 : ops[v - d.n_in].level; };
    for (uint32_t q = 0; q < d.n_ins; ++q) {
        const uint32_t w = L.ins[d.ins_off + q];
        if ((w >> 30) == INS_OP) {
            const int x = value(w & 0x3FFu), y = value((w >> 10) & 0x3FFu);
            if (x < 0 || y < 0) throw std::logic_error("dag program reads an unset accumulator");
            ops.push_back({x, y, std::max(level(x), level(y)) + 1});
            const int v = static_cast<int>(d.n_in + ops.size() - 1);
            const uint32_t rd = (w >> 20) & 0x3FFu;
            if (rd == REF_ACC)
                acc = v;
            else
                tmp[rd & 0x1FFu] = v;
        } else {
            const int v = value(w & 0x3FFu);
            if (v < 0) throw std::logic_error("dag program stores an unset accumulator");
            stores.push_back({(w >> 10) & 0xFFFFu, {v, (w >> 30) == INS_STORE_AVG}});
        }
    }
    const std::vector<int> order = dag_order(ops);
    std::map<int, std::vector<size_t>> stores_of;
    for (size_t k = 0; k < stores.size(); ++k) stores_of[stores[k].second.first].push_back(k);

    o << "__device__ __forceinline__ void dag_" << id
      << "(const KernelArgs& a, uint32_t st, uint32_t nvec, int64_t off, int ct) {\n"
         "#pragma unroll 1\n"
         "    for (uint32_t w = ct; w < 4u * nvec; w += kConsumers) {\n"
         "        const uint32_t s = st + 4u * w;\n"
         "        const int64_t pos = off + 4 * static_cast<int64_t>(w);\n";
    std::vector<char> loaded(d.n_in, 0);
    auto name = [&](int v) -> std::string {
        if (v >= static_cast<int>(d.n_in)) return "t" + std::to_string(v - d.n_in);
        if (!loaded[v]) {
            o << "        const uint32_t x" << v << " = lds32(s + " << static_cast<uint64_t>(v) * L.tile_bytes
              << "u);\n";
            loaded[v] = 1;
        }
        return "x" + std::to_string(v);
    };
    auto emit_stores = [&](int v) {
        auto it = stores_of.find(v);
        if (it == stores_of.end()) return;
        const std::string x = name(v);
        for (size_t k : it->second) {
            const uint32_t buf = stores[k].first, slot = buf >> 6, rank = buf & 63u;
            o << "        stg32(";
            if (slot == 0)
                o << "static_cast<char*>(a.bufs[" << rank << "])";
            else
                o << "(a.scratch + " << static_cast<uint64_t>(slot - 1) * P + rank << "ull * a.slot_stride)";
            o << " + pos, " << (stores[k].second.second ? "wdiv<DT>(" + x + ", " + std::to_string(P) + ".0f)" : x)
              << ");\n";
        }
    };
    for (uint32_t i = 0; i < d.n_in; ++i) emit_stores(static_cast<int>(i));
    for (int k : order) {
        const std::string x = name(ops[k].a), y = name(ops[k].b);
        o << "        const uint32_t t" << k << " = wop<DT, OP>(" << x << ", " << y << ");\n";
        emit_stores(static_cast<int>(d.n_in) + k);
    }
    o << "    }\n}\n\n";
}

}  // namespace

bool word_kernel_prefetch(const Lowered& L) {
    uint64_t ins = 0, combines = 0;
    for (uint32_t id : word_programs(L)) {
        const DevProg& d = L.progs[id];
        ins += d.n_in;
        if (d.kind == PK_DAG) {
            for (uint32_t q = 0; q < d.n_ins; ++q) combines += (L.ins[d.ins_off + q] >> 30) == INS_OP;
        } else {
            combines += d.n_in - 1;
        }
    }
    return ins > 0 && combines >= kWordPrefetchCombinesPerInput * ins;
}

int word_kernel_max_in(const Lowered& L) {
    int m = 0;
    for (uint32_t id : word_programs(L)) m = std::max<int>(m, L.progs[id].n_in);
    return m;
}

size_t word_kernel_words(const Lowered& L) {
    size_t n = 0;
    for (uint32_t id : word_programs(L)) n += L.progs[id].kind == PK_DAG ? L.progs[id].n_ins : L.progs[id].n_in;
    return n;
}

std::string word_kernel_source(const Schedule& S, const Lowered& L) {
    const std::set<uint32_t> ids = word_programs(L);
    if (ids.empty()) return std::string();
    const int op = S.op == AR_AVG ? AR_SUM : S.op;  // avg: sums, divided where stored
    const int es = esize_of(S.dtype);
    std::ostringstream o;
    o << "// word kernel of one plan: P = " << S.P << ", dtype " << S.dtype << ", op " << S.op << ", " << ids.size()
      << " programs\n"
         "typedef signed char int8_t;\ntypedef unsigned char uint8_t;\ntypedef short int16_t;\n"
         "typedef unsigned short uint16_t;\ntypedef int int32_t;\ntypedef unsigned int uint32_t;\n"
         "typedef long long int64_t;\ntypedef unsigned long long uint64_t;\n"
         "#include \"device.cuh\"\n"
         "namespace ar {\nnamespace {\n"
      << "constexpr int DT = " << S.dtype << ";\nconstexpr int OP = " << op << ";\n\n";
    const int stages = word_kernel_prefetch(L) ? word_kernel_stages(word_kernel_max_in(L)) : 0;
    for (uint32_t id : ids) emit_word_program(o, L, id, S.P, kWordThreads, stages);
    o << "}  // namespace\n}  // namespace ar\n\n"
         "extern \"C\" __global__ void __launch_bounds__("
      << kWordThreads
      << ", 1)\n"
         "ar_word_kernel(const __grid_constant__ ar::KernelArgs a) {\n"
         "    extern __shared__ __align__(128) uint8_t smem[];\n"
         "    const uint32_t sbase = ar::smem_addr(smem);\n"
         "    ar::griddep_wait();\n"
         "    ar::griddep_launch_dependents();\n"
         "    for (uint32_t it = blockIdx.x; it < a.n_items; it += gridDim.x) {\n"
         "        const ar::WorkItem w = a.items[it];\n"
         "        const int64_t off = w.elem * "
      << es
      << ";\n"
         "        const uint32_t nw = static_cast<uint32_t>((static_cast<uint64_t>(w.count) * "
      << es
      << ") >> 2);\n"
         "        switch (w.prog) {\n";
    for (uint32_t id : ids) o << "            case " << id << "u: ar::wp_" << id << "(a, off, nw, sbase); break;\n";
    o << "            default:\n"
         "                if (threadIdx.x == 0) atomicOr(a.status, ar::kStatusBadProgram);\n"
         "                return;\n"
         "        }\n"
         "    }\n"
         "}\n";
    return o.str();
}

size_t dag_kernel_words(const Lowered& L) {
    size_t n = 0;
    for (uint32_t id : staged_dag_programs(L)) n += L.progs[id].n_ins;
    return n;
}

std::string dag_kernel_source(const Schedule& S, const Lowered& L) {
    const std::set<uint32_t> ids = staged_dag_programs(L);
    if (ids.empty()) return std::string();
    const int op = S.op == AR_AVG ? AR_SUM : S.op;  // avg: sums, divided where stored
    std::ostringstream o;
    o << "// DAG kernel of one plan: P = " << S.P << ", dtype " << S.dtype << ", op " << S.op << ", "
      << ids.size() << " programs\n"
         "typedef signed char int8_t;\ntypedef unsigned char uint8_t;\ntypedef short int16_t;\n"
         "typedef unsigned short uint16_t;\ntypedef int int32_t;\ntypedef unsigned int uint32_t;\n"
         "typedef long long int64_t;\ntypedef unsigned long long uint64_t;\n"
         "#include \"device.cuh\"\n"
         "namespace ar {\nnamespace {\n"
      << "constexpr int DT = " << S.dtype << ";\nconstexpr int OP = " << op << ";\n\n";
    for (uint32_t id : ids) {
        if (L.progs[id].n_in > kWordConsumerMinIn)
            emit_program_words(o, L, id, S.P);
        else
            emit_program(o, L, id, S.P);
    }
    // The dispatch is a functor whose call operator is forced inline: as a
    // lambda, a dispatch over many programs was compiled as a called
    // function, which reached the kernel parameters through a pointer and
    // reloaded an output's buffer address from memory after every store.
    o << "struct Dispatch {\n"
         "    const KernelArgs& a;\n"
         "    __device__ __forceinline__ void operator()(const Stage& sm, const DevProg& pg, uint32_t prog,\n"
         "                                               uint32_t st, uint32_t nvec, int64_t off, int ct) const {\n"
         "        switch (prog) {\n";
    for (uint32_t id : ids) o << "            case " << id << "u: dag_" << id << "(a, st, nvec, off, ct); break;\n";
    o << "            default: dag_item<DT, OP>(a, pg, st, sm.tmps, nvec, off, ct);\n"
         "        }\n"
         "    }\n"
         "};\n\n"
         "}  // namespace\n}  // namespace ar\n\n"
         "extern \"C\" __global__ void __launch_bounds__(ar::kStagedThreads, 1)\n"
         "ar_dag_kernel(const __grid_constant__ ar::KernelArgs a) {\n"
         "    extern __shared__ __align__(128) uint8_t smem[];\n"
         "    ar::staged_body<ar::DT, ar::OP>(a, smem, ar::Dispatch{a});\n"
         "}\n";
    return o.str();
}

// ------------------------------------------------------------------ NVRTC

namespace {

// The few NVRTC entry points used, resolved from libnvrtc at run time.
struct Nvrtc {
    using Prog = void*;
    int (*create)(Prog*, const char*, const char*, int, const char* const*, const char* const*) = nullptr;
    int (*compile)(Prog, int, const char* const*) = nullptr;
    int (*cubin_size)(Prog, size_t*) = nullptr;
    int (*cubin)(Prog, char*) = nullptr;
    int (*log_size)(Prog, size_t*) = nullptr;
    int (*log)(Prog, char*) = nullptr;
    int (*destroy)(Prog*) = nullptr;
    bool ok = false;
};

const Nvrtc& nvrtc() {
    static Nvrtc n;
    static std::once_flag once;
    std::call_once(once, [] {
        const char* names[] = {"libnvrtc.so.13", "libnvrtc.so", "/usr/local/cuda/lib64/libnvrtc.so.13",
                               "/usr/local/cuda/lib64/libnvrtc.so"};
        void* h = nullptr;
        for (const char* nm : names)
            if ((h = dlopen(nm, RTLD_NOW | RTLD_LOCAL)) != nullptr) break;
        if (!h) return;
        n.create = reinterpret_cast<decltype(n.create)>(dlsym(h, "nvrtcCreateProgram"));
        n.compile = reinterpret_cast<decltype(n.compile)>(dlsym(h, "nvrtcCompileProgram"));
        n.cubin_size = reinterpret_cast<decltype(n.cubin_size)>(dlsym(h, "nvrtcGetCUBINSize"));
        n.cubin = reinterpret_cast<decltype(n.cubin)>(dlsym(h, "nvrtcGetCUBIN"));
        n.log_size = reinterpret_cast<decltype(n.log_size)>(dlsym(h, "nvrtcGetProgramLogSize"));
        n.log = reinterpret_cast<decltype(n.log)>(dlsym(h, "nvrtcGetProgramLog"));
        n.destroy = reinterpret_cast<decltype(n.destroy)>(dlsym(h, "nvrtcDestroyProgram"));
        n.ok = n.create && n.compile && n.cubin_size && n.cubin && n.log_size && n.log && n.destroy;
    });
    return n;
}

}  // namespace

bool jit_available() { return nvrtc().ok; }

int compile_dag_kernel(const std::string& src, std::string& cubin, std::string* log) {
    const Nvrtc& n = nvrtc();
    if (!n.ok) return 1;
    Nvrtc::Prog prog = nullptr;
    if (n.create(&prog, src.c_str(), "ar_dag_kernel.cu", kJitHeaderCount, kJitHeaders, kJitHeaderNames) != 0)
        return 2;
    // the same arithmetic flags as the compiled kernels: no contraction, no
    // flushing, IEEE division; unannotated (host API) declarations of ar.h
    // are taken as device declarations and never used
    const char* opts[] = {"--gpu-architecture=sm_103a", "-std=c++17", "-default-device", "--fmad=false",
                          "--ftz=false", "--prec-div=true", "--prec-sqrt=true", "-lineinfo"};
    const int rc = n.compile(prog, static_cast<int>(sizeof(opts) / sizeof(opts[0])), opts);
    if (log) {
        size_t ls = 0;
        if (n.log_size(prog, &ls) == 0 && ls > 1) {
            std::string text(ls, '\0');
            if (n.log(prog, &text[0]) == 0) *log = text.c_str();
        }
    }
    int status = 2;
    size_t cs = 0;
    if (rc == 0 && n.cubin_size(prog, &cs) == 0 && cs > 0) {
        cubin.assign(cs, '\0');
        if (n.cubin(prog, &cubin[0]) == 0) status = 0;
    }
    n.destroy(&prog);
    return status;
}

const void* load_dag_kernel(const std::string& src, const char* name) {
    static std::mutex mu;
    static std::map<std::pair<int, std::string>, const void*> cache;  // (device, source) -> kernel
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    auto key = std::make_pair(dev, src);
    auto it = cache.find(key);
    if (it != cache.end()) return it->second;
    const void* fn = nullptr;
    std::string cubin;
    if (compile_dag_kernel(src, cubin, nullptr) == 0) {
        cudaLibrary_t lib = nullptr;
        cudaKernel_t k = nullptr;
        int optin = 0;
        // the library stays loaded for the life of the process (shared by
        // every plan with the same programs)
        if (cudaLibraryLoadData(&lib, cubin.data(), nullptr, nullptr, 0, nullptr, nullptr, 0) == cudaSuccess &&
            cudaLibraryGetKernel(&k, lib, name) == cudaSuccess &&
            cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) == cudaSuccess &&
            cudaFuncSetAttribute(reinterpret_cast<const void*>(k), cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 optin) == cudaSuccess)
            fn = reinterpret_cast<const void*>(k);
    }
    cudaGetLastError();  // a failed load leaves no sticky error behind
    cache.emplace(std::move(key), fn);
    return fn;
}

}  // namespace ar
