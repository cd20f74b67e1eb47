// fast.cu -- tcgen05 tensor-core path (not yet enabled: every problem takes the SIMT path).
#include "fast.h"

bool fast_supported(const MMParams&, bool, int) { return false; }
size_t fast_scratch_bytes(const MMParams&, int) { return 0; }
cudaError_t fast_fwd(const MMParams&, const GenericPtrs&, char*, cudaStream_t) { return cudaErrorNotSupported; }
cudaError_t fast_bwd(const MMParams&, const GenericPtrs&, char*, cudaStream_t) { return cudaErrorNotSupported; }
int fastk_chunk() { return 64; }
