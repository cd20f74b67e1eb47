// rot_sincos.cuh -- sin and cos of a rotation angle, for the per-token cos / sin tables of the
// tensor-core forward.
#pragma once
#include <cuda_runtime.h>

// Cody and Waite's additive range reduction by 2 pi: k = rint(x / (2 pi)), r = (x - k P1) - k P2
// with 2 pi = P1 + P2, P1 = 201/32 (eight significant bits, so k P1 is exact for |k| < 2^16, i.e.
// |x| below about 4e5) and P2 the float nearest 2 pi - P1; then the hardware sin / cos
// approximations on r in [-pi, pi].  Absolute error a few 1e-7 for the angles the tables see
// (a GPU test checks it against sincosf).
__device__ __forceinline__ void rot_sincos(float x, float* s, float* c) {
    const float k = rintf(x * 0.159154943091895336f);  // 1 / (2 pi)
    float r = fmaf(-k, 6.28125f, x);                      // P1 = 201 / 32
    r = fmaf(-k, 1.93530717958647692e-3f, r);             // P2 = 2 pi - 201/32
    __sincosf(r, s, c);
}
