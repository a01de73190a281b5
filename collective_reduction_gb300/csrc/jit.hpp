// Run-time compiled DAG kernels.
//
// The staged kernel interprets a DAG program instruction by instruction,
// keeping temporaries in shared memory; for rank-specific results that is
// bound by instruction issue, not by HBM.  For a plan whose staged launches
// run DAG programs, this module writes the same kernel with every such
// program turned into straight-line CUDA C (temporaries become registers,
// buffer addresses and tile offsets constants), compiles it for sm_103a with
// NVRTC (loaded at run time, so the library does not depend on it) and loads
// it with the CUDA runtime.  The arithmetic is the interpreter's, in the
// interpreter's order: the results are bit for bit the same.
//
// Sets whose DAG programs read many inputs run instead on the word kernel,
// written here too: each thread takes one 32-bit word of every input
// buffer straight from global memory into registers, evaluates the item's
// program on them (chains and DAG programs alike) and stores one word to
// every output, so its footprint does not depend on the input count.
#pragma once

#include <cstddef>
#include <cstdint>
#include <string>

#include "lower.hpp"
#include "schedule.hpp"

namespace ar {

// DAG instruction words the plan's staged launches would turn into code
// (0: nothing to compile).
size_t dag_kernel_words(const Lowered& L);

// CUDA C source of the plan's DAG kernel (its entry point is
// ar_dag_kernel); empty when dag_kernel_words(L) is 0.
std::string dag_kernel_source(const Schedule& S, const Lowered& L);

// Compiles a DAG kernel source to a cubin for sm_103a.  Returns 0 on
// success, 1 if NVRTC cannot be loaded, 2 if the compilation failed (the
// compiler's log in *log when log is not null).
int compile_dag_kernel(const std::string& src, std::string& cubin, std::string* log);

// Instruction words of the programs the plan's word-kernel launches run
// (0: no word-kernel launch).
size_t word_kernel_words(const Lowered& L);

// Most inputs of a program of the plan's word-kernel launches (0: none).
int word_kernel_max_in(const Lowered& L);

// Whether the plan's word kernel prefetches input words through shared
// memory (its programs average at least kWordPrefetchCombinesPerInput
// combines per input: long enough evaluations to hide the next position's
// loads behind; measured 3-9 points faster at P = 63 / 64 with 6-10 per input,
// 3-9 points slower at P = 48 / 63 with 1-4 per input).  Its dynamic shared
// memory is then word_kernel_smem(word_kernel_max_in(L)), else none.
constexpr uint64_t kWordPrefetchCombinesPerInput = 5;
bool word_kernel_prefetch(const Lowered& L);

// CUDA C source of the plan's word kernel (its entry point is
// ar_word_kernel); empty when word_kernel_words(L) is 0.
std::string word_kernel_source(const Schedule& S, const Lowered& L);

// True when NVRTC can be loaded (the run-time compiled kernels are possible).
bool jit_available();

// The loaded kernel `name` of src on the current device (compiled and loaded
// once per source and device, then cached), ready for cudaLaunchKernel with
// the dynamic shared memory limit raised; nullptr on any failure.
const void* load_dag_kernel(const std::string& src, const char* name = "ar_dag_kernel");

}  // namespace ar
