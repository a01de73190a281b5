// Kernel launch interface between the C ABI and the CUDA kernels.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

#include "kargs.hpp"

namespace ar {

// Launches kernel f (one KernelArgs parameter) as a programmatic dependent
// of the previous kernel in the stream (see device.cuh).
cudaError_t launch_dependent(const void* f, int grid, int block, int smem, cudaStream_t st, const KernelArgs& a);
// One CTA that waits on an mbarrier nothing completes, bounded by ns.
cudaError_t launch_wait_selftest(int* status, uint64_t ns, cudaStream_t st);
// Sets the dynamic shared-memory limits of the (dtype, op) kernels.
cudaError_t prepare_kernels(int dtype, int op);
// Persistent staged kernel over a.items (all 16-byte aligned), grid CTAs.
cudaError_t launch_staged(int dtype, int op, const KernelArgs& a, int grid, int smem, cudaStream_t st);
// Persistent rank-streaming kernel over a.items (chain / FP32ACC programs only).
cudaError_t launch_stream(int dtype, int op, const KernelArgs& a, int grid, int smem, cudaStream_t st);
// Chain programs of at most max_in inputs, 32-bit words of every input in
// registers (kChainWordThreads per CTA, grid CTAs over a.items; a persistent
// grid is kChainWordCtasPerSm CTAs per SM).
constexpr int kChainWordCtasPerSm = 4;
cudaError_t launch_chain_words(int dtype, int op, const KernelArgs& a, int max_in, int grid, cudaStream_t st);
// One CTA per item, one element per thread.
cudaError_t launch_elementwise(int dtype, int op, const KernelArgs& a, int smem, cudaStream_t st);
// The copy kernel over a.items (programs of one input: copies to every
// output), kCopyThreads per CTA, grid CTAs (a CTA takes items blockIdx.x,
// + grid, ...); any dtype and op (nothing is combined).  Launched with up to
// kCopyCtasPerSm CTAs per SM, in practice one per item: the hardware deals
// them to the SMs as earlier ones finish.
#ifndef AR_COPY_CTAS_PER_SM
#define AR_COPY_CTAS_PER_SM 1024
#endif
constexpr int kCopyCtasPerSm = AR_COPY_CTAS_PER_SM;
cudaError_t launch_copies(int dtype, const KernelArgs& a, int grid, cudaStream_t st);
// The few-input kernel over a.items (chains and fp32 accumulations of at
// most kFewMaxIn inputs, or with `trees` chains and single trees of at most
// kFewTreeMaxIn; max_in: the most of the launch's programs), the copy
// kernel's grid shape.
cudaError_t launch_few(int dtype, int op, const KernelArgs& a, int max_in, bool trees, int grid, cudaStream_t st);

}  // namespace ar
