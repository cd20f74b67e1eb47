// finite.h -- host entry of the optional output finiteness check (finite.cu).
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

// Up to seven device buffers (the outputs of one call), checked in one launch.
struct FiniteSegs {
    int n;
    const void* ptr[7];
    int64_t bytes[7];
    int bf16[7];  // 1: elements are bf16, else fp32
};

// Enqueues the check on `st`; sets *flag (device int, not cleared here) to 1 if any element of
// any buffer is NaN or infinite.
cudaError_t launch_finite_check(const FiniteSegs& segs, int* flag, cudaStream_t st);
