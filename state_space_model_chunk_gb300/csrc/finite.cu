// finite.cu -- the optional output check (MM_FLAG_CHECK_FINITE): one pass over the outputs of a
// call that raises a flag word in the workspace header if any element is NaN or infinite.
//
// burn-mamba, "mamba3/moments/recalculated.rs", moments_phys_fwd: after the chunk loop the pages
// pass (m2, m1) through `san`, a sanity hook whose body is not shown.  Read here as a finiteness
// check of the results that does not change them; the backward's gradients get the same check.
#include <cuda_runtime.h>
#include <stdint.h>

#include "finite.h"
#include "prof.h"

namespace {

// Exponent field all ones <=> NaN or infinity.
__device__ __forceinline__ bool bad_f32(uint32_t w) { return (w & 0x7F800000u) == 0x7F800000u; }
__device__ __forceinline__ bool bad_bf16x2(uint32_t w) {
    return (w & 0x7F80u) == 0x7F80u || (w & 0x7F800000u) == 0x7F800000u;
}

__global__ void k_check_finite(FiniteSegs segs, int* flag) {
    bool bad = false;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    for (int s = 0; s < segs.n; ++s) {
        const unsigned char* base = static_cast<const unsigned char*>(segs.ptr[s]);
        const int64_t bytes = segs.bytes[s];
        const bool bf16 = segs.bf16[s] != 0;
        const int64_t nvec = bytes >> 4;  // 16-byte pieces (every tensor starts 16-byte aligned)
        for (int64_t i = tid; i < nvec; i += stride) {
            const uint4 v = reinterpret_cast<const uint4*>(base)[i];
            if (bf16)
                bad |= bad_bf16x2(v.x) | bad_bf16x2(v.y) | bad_bf16x2(v.z) | bad_bf16x2(v.w);
            else
                bad |= bad_f32(v.x) | bad_f32(v.y) | bad_f32(v.z) | bad_f32(v.w);
        }
        // the ragged end: whole elements past the last 16-byte piece
        const int64_t tail0 = nvec << 4;
        const int64_t esz = bf16 ? 2 : 4;
        for (int64_t i = tail0 / esz + tid; i < bytes / esz; i += stride) {
            if (bf16) {
                const uint16_t h = reinterpret_cast<const uint16_t*>(base)[i];
                bad |= (h & 0x7F80u) == 0x7F80u;
            } else {
                bad |= bad_f32(reinterpret_cast<const uint32_t*>(base)[i]);
            }
        }
    }
    if (__any_sync(0xffffffffu, bad) && (threadIdx.x & 31) == 0) atomicOr(flag, 1);
}

}  // namespace

cudaError_t launch_finite_check(const FiniteSegs& segs, int* flag, cudaStream_t st) {
    if (segs.n == 0) return cudaSuccess;
    int64_t vec = 0;
    for (int s = 0; s < segs.n; ++s) vec += segs.bytes[s] >> 4;
    int grid = (int)((vec + 255) / 256);
    if (grid < 1) grid = 1;
    if (grid > 4 * 152) grid = 4 * 152;  // a few waves of 256-thread blocks over the 152 SMs
    mm_prof_mark(KID_FINITE, 1, st);
    k_check_finite<<<grid, 256, 0, st>>>(segs, flag);
    mm_prof_mark(KID_FINITE, 0, st);
    return cudaGetLastError();
}
