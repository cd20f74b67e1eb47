// common.cuh -- device-side problem description and small helpers shared by the kernels
// of libmoments.so (SIMT and tensor-core paths).
#pragma once
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#define MM_MAX_B 512  // batch rows whose valid lengths travel in the kernel parameters

enum { ROT_NONE = 0, ROT_PAIRWISE = 1, ROT_HALF = 2, ROT_QUAT = 3 };

// Everything a kernel needs to know about the problem, passed by value.
struct MMParams {
    int b, s, C, h, p, r, l, nc;  // nc = s / l chunks per row
    int rot;                      // ROT_*
    int na;                       // complex kinds: angles per token (rope_dim / 2); else 0
    int J;                        // quaternion blocks; else 0
    int rw;                       // floats of rot per (b, t, h): na or 4 J
    // The tensor-core path splits a head's p state rows into `groups` groups of 64 rows and runs
    // each group as a head of its own: h = heads * groups and p = 64 there, so that tensors
    // indexed by state row (xhat, states, carries, d_xhat, d_initial) keep their layout, while the
    // tensors shared by a head's rows (bhat, da, rot and their gradients, d_m2, d_m1) are indexed
    // by the caller's head, h / groups.  Outside that path groups = 1 and heads = h.
    int heads;
    int groups;
    // Rows of xhat / d_xhat per (row-group) head in the caller's layout: p, except on the
    // tensor-core path for p below 64, where the kernels run 64 rows (p = 64) and the rows past
    // prow are zero.
    int prow;
    int valid[MM_MAX_B];          // valid_len per batch row, clamped to [0, s]
};

__host__ __device__ inline int mm_processed(const MMParams& P, int bb) {
    // chunks whose start lies before valid_len ("processed" of the recompute backward)
    int v = P.valid[bb];
    int pc = (v + P.l - 1) / P.l;
    return pc < P.nc ? pc : P.nc;
}
__host__ __device__ inline int mm_chunk_rows(const MMParams& P, int bb, int n) {
    // valid tokens of chunk n in row bb ("chunk_mask": saturating start, min chunk_len)
    int v = P.valid[bb] - n * P.l;
    return v < 0 ? 0 : (v > P.l ? P.l : v);
}

// Row-major offsets.
__device__ __forceinline__ int64_t off_x(const MMParams& P, int bb, int t, int c, int hh) {
    return ((((int64_t)bb * P.s + t) * P.C + c) * P.h + hh) * P.prow;
}
// bhat / da / rot and their gradients: hh is the caller's head (see MMParams::heads)
__device__ __forceinline__ int64_t off_b(const MMParams& P, int bb, int t, int c, int hh) {
    return ((((int64_t)bb * P.s + t) * P.C + c) * P.heads + hh) * P.r;
}
__device__ __forceinline__ int64_t off_da(const MMParams& P, int bb, int t, int hh) {
    return ((int64_t)bb * P.s + t) * P.heads + hh;
}
__device__ __forceinline__ int64_t off_rot(const MMParams& P, int bb, int t, int hh) {
    return (((int64_t)bb * P.s + t) * P.heads + hh) * P.rw;
}
// [b, h, nc, p, r] carries / cotangent carries
__device__ __forceinline__ int64_t off_carry(const MMParams& P, int bb, int hh, int n) {
    return (((int64_t)bb * P.h + hh) * P.nc + n) * ((int64_t)P.p * P.r);
}

__device__ __forceinline__ float ld_val(const float* p) { return *p; }
__device__ __forceinline__ float ld_val(const __nv_bfloat16* p) { return __bfloat162float(*p); }
__device__ __forceinline__ void st_val(float* p, float v) { *p = v; }
__device__ __forceinline__ void st_val(__nv_bfloat16* p, float v) { *p = __float2bfloat16_rn(v); }

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Sum over the block; every thread gets the result.  `red` holds >= 32 floats.
__device__ __forceinline__ float block_sum(float v, float* red) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = (blockDim.x + 31) >> 5;
    v = warp_sum(v);
    __syncthreads();
    if (lane == 0) red[wid] = v;
    __syncthreads();
    float t = (threadIdx.x < (unsigned)nw) ? red[threadIdx.x] : 0.f;
    if (wid == 0) t = warp_sum(t);
    if (threadIdx.x == 0) red[0] = t;
    __syncthreads();
    float out = red[0];
    __syncthreads();
    return out;
}
