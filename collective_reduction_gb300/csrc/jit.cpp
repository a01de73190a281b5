// Run-time compiled DAG kernels: source generation, NVRTC compilation and
// loading (see jit.hpp).
#include "jit.hpp"

#include <cuda_runtime.h>
#include <dlfcn.h>

#include <cstdio>
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
        if (s.stream || s.small) continue;
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

}  // namespace

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
    for (uint32_t id : ids) emit_program(o, L, id, S.P);
    o << "}  // namespace\n}  // namespace ar\n\n"
         "extern \"C\" __global__ void __launch_bounds__(ar::kStagedThreads, 1)\n"
         "ar_dag_kernel(const __grid_constant__ ar::KernelArgs a) {\n"
         "    extern __shared__ __align__(128) uint8_t smem[];\n"
         "    ar::staged_body<ar::DT, ar::OP>(a, smem, [&](const ar::Stage& sm, const ar::DevProg& pg, uint32_t prog,\n"
         "                                              uint32_t st, uint32_t nvec, int64_t off, int ct) {\n"
         "        switch (prog) {\n";
    for (uint32_t id : ids) o << "            case " << id << "u: ar::dag_" << id << "(a, st, nvec, off, ct); break;\n";
    o << "            default: ar::dag_item<ar::DT, ar::OP>(a, pg, st, sm.tmps, nvec, off, ct);\n"
         "        }\n"
         "    });\n"
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

const void* load_dag_kernel(const std::string& src) {
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
            cudaLibraryGetKernel(&k, lib, "ar_dag_kernel") == cudaSuccess &&
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
