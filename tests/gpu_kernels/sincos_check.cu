// Test kernel: rot_sincos (the forward's table routine) next to sincosf on the same angles.
#include "../../state_space_model_chunk_gb300/csrc/rot_sincos.cuh"

__global__ void sincos_check_kernel(const float* x, float* out, int n) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    float s, c, s0, c0;
    rot_sincos(x[i], &s, &c);
    sincosf(x[i], &s0, &c0);
    out[4 * i + 0] = s;
    out[4 * i + 1] = c;
    out[4 * i + 2] = s0;
    out[4 * i + 3] = c0;
}

extern "C" int sincos_check(const float* x, float* out, int n) {
    if (n <= 0) return 0;
    sincos_check_kernel<<<(n + 255) / 256, 256>>>(x, out, n);
    return (int)cudaDeviceSynchronize();
}
