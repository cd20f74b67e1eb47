// rot_steps.h -- the cumulative rotation built from per-token steps (MM_FLAG_ROT_STEPS) and the
// gradient of that build; see rot_steps.cu.
#pragma once
#include <cuda_runtime.h>

#include "common.cuh"

// Scratch the two passes below need (one float per row, 64-token chunk and angle column; two
// float4 per row, chunk and quaternion).
size_t rot_steps_scratch_bytes(const MMParams& P);
// cum = the cumulative rotation of `steps` (both [b, s, h, rw] fp32, 16-byte aligned).
cudaError_t rot_steps_build(const MMParams& P, const float* steps, float* cum, void* scratch, cudaStream_t st);
// d_steps = the gradient w.r.t. `steps`, given d_cum, the gradient w.r.t. cum = build(steps).
cudaError_t rot_steps_vjp(const MMParams& P, const float* steps, const float* cum, const float* d_cum, float* d_steps,
                          void* scratch, cudaStream_t st);
