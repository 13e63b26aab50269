// Allocation-free variant of the bf16 GEMM entry point.
//
// Some callers cannot allocate device memory at the point where they want to
// run a projection: code running inside another framework's memory pool that
// forbids raw cudaMalloc, real-time paths where an allocation (and the device
// synchronisation it can imply) is not allowed, or plug-ins that must not grow
// the process's footprint after start-up.  For them this variant keeps its
// split-K scratch (the fp32 partial tiles that several CTAs leave for the
// fixup kernel) in a fixed array that lives in the library's module for the
// whole life of the process, instead of in a caller-provided workspace.
#pragma once
#include <cuda_runtime.h>

#include "gemm_tc.cuh"

namespace dinfer {

// Limits of the fixed scratch: token rows M <= 64 (one 64-token tile), at most
// kNoAllocMaxCtas CTAs, each leaving at most two partial 128 x 64 fp32 tiles.
constexpr int kNoAllocMaxRows = 64;
constexpr int kNoAllocMaxCtas = 152;
constexpr size_t kNoAllocScratchFloats = (size_t)kNoAllocMaxCtas * 2 * 64 * 128;  // 9.5 MiB

// One copy per GPU that loads the library, held until the process exits.
// Every call shares it: calls that overlap on the GPU (different streams, or
// several host threads) race on it and must be serialised by the caller.
static __device__ __align__(256) float g_noalloc_scratch[kNoAllocScratchFloats];
// Device status word written by the kernels (pipeline wait timeouts).
static __device__ __align__(256) DevState g_noalloc_state;

}  // namespace dinfer
