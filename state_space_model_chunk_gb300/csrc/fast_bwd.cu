// fast_bwd.cu -- host side of the tcgen05 recompute backward (the kernel itself:
// fast_bwd_kernel.cuh), and the pass that finishes d_rot from the kernel's partial sums.
#include "fast_bwd_kernel.cuh"

namespace fastbwd {

// d_rot = (sum over rows 0-31) + (sum over rows 32-63) of every valid token, in that order: the
// two row warps of a chunk store their partial sums with plain stores, one into d_rot and one into
// the workspace, and this pass adds them (no atomics, and a result that does not depend on
// timing); drot2 null: d_rot already holds the sum.  Quaternions (rot not null): the summed
// sum_p d_c (x) conj(c) of each block times Q / |Q|^2, Q the block's cumulative quaternion.  One
// float4 (a quaternion block) per thread; rows past valid_len keep the zeros the host wrote.
__global__ void __launch_bounds__(256) k_drot_finish(const __grid_constant__ MMParams P, float* __restrict__ drot,
                                                     const float* __restrict__ drot2, const float* __restrict__ rot,
                                                     int64_t n4) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n4) return;
    const int64_t row = i / (P.rw >> 2);  // (bb, t, hh)
    const int64_t bt = row / P.heads;
    const int bb = (int)(bt / P.s), t = (int)(bt - (int64_t)bb * P.s);
    if (t >= P.valid[bb]) return;
    float4 a = reinterpret_cast<float4*>(drot)[i];
    if (drot2) {
        const float4 c = reinterpret_cast<const float4*>(drot2)[i];
        a.x += c.x; a.y += c.y; a.z += c.z; a.w += c.w;
    }
    if (rot) {
        const float4 q = reinterpret_cast<const float4*>(rot)[i];
        float o0, o1, o2, o3;
        hamilton(a.x, a.y, a.z, a.w, q.x, q.y, q.z, q.w, o0, o1, o2, o3);
        const float inv = 1.f / (q.x * q.x + q.y * q.y + q.z * q.z + q.w * q.w);
        a = make_float4(inv * o0, inv * o1, inv * o2, inv * o3);
    }
    reinterpret_cast<float4*>(drot)[i] = a;
}

}  // namespace fastbwd

// ----------------------------------------------------------------------------- host side
namespace fastk {

size_t bwd_anchor_bytes() { return (size_t)kMaxBwdGrid * fastbwd::NANCHOR * 128 * 128 * sizeof(float); }
size_t bwd_drot2_bytes(const MMParams& P) { return (size_t)P.b * P.s * P.heads * P.rw * sizeof(float); }

cudaError_t launch_tc_bwd(const FastArgs& fa, float* E, float* anchors, float* drot2, const float* dm2, const float* dm1,
                          void* dx, void* db, float* dda, float* drot, const float* rot, const TensorMaps& maps, int grid,
                          cudaStream_t st) {
    using namespace fastbwd;
    BwdArgs a;
    a.F = fa;
    a.E = E;
    a.anchors = anchors;
    a.dm2 = dm2;
    a.dm1 = dm1;
    a.dx = static_cast<__nv_bfloat16*>(dx);
    a.db = static_cast<__nv_bfloat16*>(db);
    a.dda = dda;
    a.drot = drot;
    a.drot2 = drot2;
    const int64_t ntok = (int64_t)fa.P.b * fa.P.s;
    const bool grouped = fa.P.groups > 1;
    a.db_slice = grouped ? ntok * fa.P.C * fa.P.heads * fa.P.r : 0;
    a.dda_slice = grouped ? ntok * fa.P.heads : 0;
    a.drot_slice = grouped ? ntok * fa.P.heads * fa.P.rw : 0;
    // channel slots per chunk in the span tiles: 4 when C <= 4, else 8
    decltype(&tc_bwd_kernel<ROT_NONE, 0, 2, false>) kern;
    // (the general-shape instantiations: a partial last chunk, or fewer than 64 rows per head)
    const bool c8 = fa.P.C > 4, rag = (fa.P.s % FL) != 0 || fa.P.prow < fa.P.p;
#define BWD_KERN(K, L) (c8 ? tc_bwd_kernel<K, L, 3, false> : tc_bwd_kernel<K, L, 2, false>)
    switch (fa.P.rot) {
        case ROT_PAIRWISE: kern = BWD_KERN(ROT_PAIRWISE, 0); break;
        case ROT_HALF: kern = fa.layoutB ? BWD_KERN(ROT_HALF, 1) : BWD_KERN(ROT_HALF, 0); break;
        case ROT_QUAT: kern = BWD_KERN(ROT_QUAT, 0); break;
        default: kern = BWD_KERN(ROT_NONE, 0); break;
    }
#undef BWD_KERN
    if (rag) kern = ragged_bwd_kernel(fa.P.rot, fa.layoutB, c8);
    cudaError_t e = mm_allow_smem(reinterpret_cast<const void*>(kern), (int)SMEM_BYTES);
    if (e != cudaSuccess) return e;
    mm_prof_mark(KID_FAST_BWD, 1, st);
    kern<<<grid, NTHR, SMEM_BYTES, st>>>(a, maps.x, maps.b, maps.rot, maps.da64);
    mm_prof_mark(KID_FAST_BWD, 0, st);
    if ((e = cudaGetLastError()) != cudaSuccess || fa.P.rw == 0) return e;
    // with row groups the per-group slices are summed by the caller, which then finishes d_rot
    if (fa.P.groups > 1) return e;
    return launch_drot_finish(fa.P, drot, drot2, rot, st);
}

cudaError_t launch_drot_finish(const MMParams& P, float* drot, const float* drot2, const float* rot, cudaStream_t st) {
    using namespace fastbwd;
    if (P.rw == 0 || (!drot2 && P.rot != ROT_QUAT)) return cudaSuccess;
    const int64_t n4 = (int64_t)P.b * P.s * P.heads * (P.rw >> 2);
    mm_prof_mark(KID_DROT_SUM, 1, st);
    k_drot_finish<<<(unsigned)((n4 + 255) / 256), 256, 0, st>>>(P, drot, drot2, P.rot == ROT_QUAT ? rot : nullptr, n4);
    mm_prof_mark(KID_DROT_SUM, 0, st);
    return cudaGetLastError();
}

}  // namespace fastk
