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

// The loaded kernel for src on the current device (compiled and loaded once
// per source and device, then cached), ready for cudaLaunchKernel with the
// dynamic shared memory limit raised; nullptr on any failure.
const void* load_dag_kernel(const std::string& src);

}  // namespace ar
