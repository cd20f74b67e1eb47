// fast.h -- host entry points of the tcgen05 tensor-core path (fast_fwd.cu / fast_bwd.cu).
#pragma once
#include "common.cuh"
#include "generic.h"

// Whether the tensor-core kernels implement this problem (bf16 operands and the tile shapes
// they are built for); otherwise the SIMT kernels run.
bool fast_supported(const MMParams& P, bool bf16, int backward);
size_t fast_scratch_bytes(const MMParams& P, int backward);
cudaError_t fast_fwd(const MMParams& P, const GenericPtrs& A, char* scratch, cudaStream_t st);
cudaError_t fast_bwd(const MMParams& P, const GenericPtrs& A, char* scratch, cudaStream_t st);
int fastk_chunk();  // internal chunk length of the tensor-core path
