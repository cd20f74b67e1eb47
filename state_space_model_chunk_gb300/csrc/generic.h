// generic.h -- host entry points of the SIMT fp32 kernels (generic.cu).
#pragma once
#include "common.cuh"

struct GenericPtrs {
    int reuse_carries;  // backward: Hc / Dn already hold this problem's carries (from its forward)
    int test_wait_timeout;  // forward, tensor-core path: MM_FLAG_TEST_WAIT_TIMEOUT
    const void* xhat;
    const void* bhat;
    const float* da;
    const float* rot;
    const float* initial;
    float* m2;
    float* m1;
    const float* dm2;
    const float* dm1;
    void* dxhat;
    void* dbhat;
    float* dda;
    float* drot;
    float* dinit;
    // workspace carve-outs
    float* Hc;    // [b,h,nc,p,r] carries
    float* Dn;    // [b,h,nc] chunk decays
    float* E;     // [b,h,nc,p,r] carry cotangents
    float* dsym;  // [b,h,r,r] d_m2 + d_m2^T
    float* traj;  // [grid, l, p, r] per-block chunk state scratch
    int* err;     // device error word (tensor-core path)
};

size_t generic_fwd_smem(const MMParams& P);
size_t generic_bwd_smem(const MMParams& P);
size_t generic_correct_smem(const MMParams& P);
size_t generic_end_smem(const MMParams& P);
bool generic_supported(const MMParams& P, int smem_limit);
cudaError_t generic_fwd(const MMParams& P, bool bf16, const GenericPtrs& A, cudaStream_t st);
cudaError_t generic_bwd(const MMParams& P, bool bf16, const GenericPtrs& A, int grid, cudaStream_t st);
cudaError_t generic_carry_scan(const MMParams& P, const float* initial, float* Hc, const float* Dn,
                               cudaStream_t st);
cudaError_t generic_cot_scan(const MMParams& P, float* E, const float* Dn, float* dinit, cudaStream_t st);
cudaError_t generic_dsym(const MMParams& P, const float* dm2, float* dsym, cudaStream_t st);
