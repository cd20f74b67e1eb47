// fast.cu -- host side of the tcgen05 path: eligibility, tensor-map encoding, dispatch.
#include <cuda.h>

#include <cstring>

#include "fast.h"
#include "fast_common.cuh"
#include "generic.h"

namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static bool tried = false;
    if (!tried) {
        tried = true;
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
        else
            cudaGetLastError();
    }
    return fn;
}

cudaError_t encode(CUtensorMap* m, CUtensorMapDataType dt, cuuint32_t rank, const void* base, const cuuint64_t* dims,
                   const cuuint64_t* strides, const cuuint32_t* box, CUtensorMapSwizzle sw) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return cudaErrorNotSupported;
    cuuint32_t es[5] = {1, 1, 1, 1, 1};
    CUresult r = fn(m, dt, rank, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

MMParams internal_params(const MMParams& P0) {
    MMParams P = P0;
    P.l = fastk::FL;
    P.nc = P.s / fastk::FL;
    return P;
}

}  // namespace

namespace fastk {

int sm_count() {
    static int n = 0;
    if (!n) {
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            cudaGetLastError();
            n = 148;
        }
    }
    return n;
}

cudaError_t encode_grad_maps(const MMParams& P, const void* dx, const void* db, TensorMaps* maps) {
    const cuuint64_t bs = (cuuint64_t)P.b * P.s;
    cudaError_t e;
    {   // as x32, over d_xhat
        cuuint64_t dims[4] = {(cuuint64_t)P.p, (cuuint64_t)P.h, (cuuint64_t)P.C, bs};
        cuuint64_t str[3] = {(cuuint64_t)P.p * 2, (cuuint64_t)P.h * P.p * 2, (cuuint64_t)P.C * P.h * P.p * 2};
        cuuint32_t box[4] = {64, 1, (cuuint32_t)P.C, (cuuint32_t)corr_tps(P)};
        if ((e = encode(&maps->dx32, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, dx, dims, str, box,
                        CU_TENSOR_MAP_SWIZZLE_128B)) != cudaSuccess)
            return e;
    }
    {   // as b32, over d_bhat (a box's columns past r are skipped by the stores)
        cuuint64_t dims[4] = {(cuuint64_t)P.r, (cuuint64_t)P.h, (cuuint64_t)P.C, bs};
        cuuint64_t str[3] = {(cuuint64_t)P.r * 2, (cuuint64_t)P.h * P.r * 2, (cuuint64_t)P.C * P.h * P.r * 2};
        cuuint32_t box[4] = {64, 1, (cuuint32_t)P.C, (cuuint32_t)corr_tps(P)};
        if ((e = encode(&maps->db32, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, db, dims, str, box,
                        CU_TENSOR_MAP_SWIZZLE_128B)) != cudaSuccess)
            return e;
    }
    return cudaSuccess;
}

cudaError_t encode_maps(const MMParams& P, const void* xhat, const void* bhat, const float* rot, const float* da,
                        TensorMaps* maps) {
    const cuuint64_t bs = (cuuint64_t)P.b * P.s;
    cudaError_t e;
    {   // xhat as [b*s, C, h, p] bf16; box = the C rows of one (token, head)
        cuuint64_t dims[4] = {(cuuint64_t)P.p, (cuuint64_t)P.h, (cuuint64_t)P.C, bs};
        cuuint64_t str[3] = {(cuuint64_t)P.p * 2, (cuuint64_t)P.h * P.p * 2, (cuuint64_t)P.C * P.h * P.p * 2};
        cuuint32_t box[4] = {64, 1, (cuuint32_t)P.C, 1};
        if ((e = encode(&maps->x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, xhat, dims, str, box,
                        CU_TENSOR_MAP_SWIZZLE_128B)) != cudaSuccess)
            return e;
        box[3] = 8;  // 8 consecutive tokens: rows (token, channel)
        if ((e = encode(&maps->x8, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, xhat, dims, str, box,
                        CU_TENSOR_MAP_SWIZZLE_128B)) != cudaSuccess)
            return e;
        box[3] = (cuuint32_t)corr_tps(P);
        if ((e = encode(&maps->x32, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, xhat, dims, str, box,
                                    CU_TENSOR_MAP_SWIZZLE_128B)) != cudaSuccess)
            return e;
    }
    {   // bhat as [b*s, C, h, r] bf16; box = 64 columns (from column 64 a) of the C rows: columns
        // past r read as zeros, so an r below 128 leaves the tiles' tail zero
        cuuint64_t dims[4] = {(cuuint64_t)P.r, (cuuint64_t)P.h, (cuuint64_t)P.C, bs};
        cuuint64_t str[3] = {(cuuint64_t)P.r * 2, (cuuint64_t)P.h * P.r * 2, (cuuint64_t)P.C * P.h * P.r * 2};
        cuuint32_t box[4] = {64, 1, (cuuint32_t)P.C, 1};
        if ((e = encode(&maps->b, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, bhat, dims, str, box,
                        CU_TENSOR_MAP_SWIZZLE_128B)) != cudaSuccess)
            return e;
        box[3] = 8;
        if ((e = encode(&maps->b8, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, bhat, dims, str, box,
                        CU_TENSOR_MAP_SWIZZLE_128B)) != cudaSuccess)
            return e;
        box[3] = (cuuint32_t)corr_tps(P);
        if ((e = encode(&maps->b32, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, bhat, dims, str, box,
                                    CU_TENSOR_MAP_SWIZZLE_128B)) != cudaSuccess)
            return e;
    }
    if (P.rw > 0) {  // rot as [b*s, h, rw] fp32; box = one (token, head)
        cuuint64_t dims[3] = {(cuuint64_t)P.rw, (cuuint64_t)P.h, bs};
        cuuint64_t str[2] = {(cuuint64_t)P.rw * 4, (cuuint64_t)P.h * P.rw * 4};
        cuuint32_t box[3] = {(cuuint32_t)P.rw, 1, 1};
        if ((e = encode(&maps->rot, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, rot, dims, str, box,
                        CU_TENSOR_MAP_SWIZZLE_NONE)) != cudaSuccess)
            return e;
    } else {
        std::memset(&maps->rot, 0, sizeof(maps->rot));
    }
    if (!da_by_tma(P)) {  // rows of h floats that are not 16-byte multiples: the kernels load da themselves
        std::memset(&maps->da, 0, sizeof(maps->da));
        std::memset(&maps->da64, 0, sizeof(maps->da64));
    } else {   // da as [b*s, h] fp32; box = 4 heads of one token (16 bytes)
        cuuint64_t dims[2] = {(cuuint64_t)P.h, bs};
        cuuint64_t str[1] = {(cuuint64_t)P.h * 4};
        cuuint32_t box[2] = {4, 1};
        if ((e = encode(&maps->da, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, da, dims, str, box,
                        CU_TENSOR_MAP_SWIZZLE_NONE)) != cudaSuccess)
            return e;
        cuuint32_t box64[2] = {4, 64};  // 4 heads x one 64-token chunk
        if ((e = encode(&maps->da64, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, da, dims, str, box64,
                        CU_TENSOR_MAP_SWIZZLE_NONE)) != cudaSuccess)
            return e;
    }
    return cudaSuccess;
}

}  // namespace fastk

int fastk_chunk() { return fastk::FL; }

bool fast_supported(const MMParams& P, bool bf16, int backward) {
    if (!bf16) return false;
    // r: a multiple of 16 up to 128 (the tiles hold 128 columns, and the columns past r load as
    // zeros); half-split pairs columns r / 2 apart, which the thread layouts hold for 64 or 128 only
    if (P.p != 64 || P.r < 16 || P.r > 128 || P.r % 16 || P.C < 1 || P.C > 8) return false;
    if (P.rot == ROT_HALF && P.r != 64 && P.r != 128) return false;
    if (P.s % fastk::FL || P.b > MM_MAX_B) return false;
    // rows of angles / quaternions are copied as 16-byte multiples, at most 128 floats
    if (P.rw % 4 || P.rw > 128) return false;
    if (!encode_fn()) return false;
    return true;
}

size_t fast_scratch_bytes(const MMParams& P, int backward) {
    if (!backward) return fastk::fwd_partial_bytes(internal_params(P));
    const size_t a = fastk::bwd_anchor_bytes();  // a multiple of 256 bytes
    return a + fastk::bwd_drot2_bytes(P);
}

cudaError_t fast_fwd(const MMParams& P0, const GenericPtrs& A, char* scratch, cudaStream_t st) {
    using namespace fastk;
    const MMParams P = internal_params(P0);
    FastArgs fa;
    std::memset(&fa, 0, sizeof(fa));
    fa.P = P;
    fa.layoutB = (P.rot == ROT_HALF && P.r == 64) ? 1 : 0;
    fa.items = count_items(P);
    fa.Hc = A.Hc;
    fa.Dn = A.Dn;
    fa.m2 = A.m2;
    fa.m1 = A.m1;
    fa.m2p = reinterpret_cast<float*>(scratch);
    fa.da = A.da;
    fa.err = A.err;
    fa.test_wait_timeout = A.test_wait_timeout;
    if (fa.items == 0) return cudaSuccess;  // nothing valid: m2 / m1 stay zero
    TensorMaps maps;
    cudaError_t e = encode_maps(P, A.xhat, A.bhat, A.rot, A.da, &maps);
    if (e != cudaSuccess) return e;
    int grid = fa.items < sm_count() ? fa.items : sm_count();
    if (grid > kMaxFwdGrid) grid = kMaxFwdGrid;
    if ((e = launch_tc_end(fa, maps, st)) != cudaSuccess) return e;
    if ((e = generic_carry_scan(P, A.initial, A.Hc, A.Dn, st)) != cudaSuccess) return e;
    return launch_tc_fwd(fa, maps, grid, st);
}

cudaError_t fast_bwd(const MMParams& P0, const GenericPtrs& A, char* scratch, cudaStream_t st) {
    using namespace fastk;
    const MMParams P = internal_params(P0);
    FastArgs fa;
    std::memset(&fa, 0, sizeof(fa));
    fa.P = P;
    fa.layoutB = (P.rot == ROT_HALF && P.r == 64) ? 1 : 0;
    fa.items = count_items(P);
    fa.Hc = A.Hc;
    fa.Dn = A.Dn;
    fa.da = A.da;
    fa.err = A.err;
    cudaError_t e;
    // d_da and d_rot start from zero: the kernels write them for valid positions only (d_rot as
    // two partial sums that a second pass adds; d_da then gets the correction added).  d_xhat / d_bhat at positions at or past valid_len are exactly zero; every
    // position before is written.
    const size_t bs = (size_t)P.b * P.s;
    if ((e = cudaMemsetAsync(A.dda, 0, sizeof(float) * bs * P.h, st)) != cudaSuccess) return e;
    if (P.rw && (e = cudaMemsetAsync(A.drot, 0, sizeof(float) * bs * P.h * P.rw, st)) != cudaSuccess) return e;
    const size_t es = 2;
    for (int bb = 0; bb < P.b; ++bb) {
        const size_t v = (size_t)P.valid[bb], tail = (size_t)P.s - v;
        if (!tail) continue;
        const size_t row0 = (size_t)bb * P.s + v;
        if ((e = cudaMemsetAsync(static_cast<char*>(A.dxhat) + es * row0 * P.C * P.h * P.p, 0,
                                 es * tail * P.C * P.h * P.p, st)) != cudaSuccess ||
            (e = cudaMemsetAsync(static_cast<char*>(A.dbhat) + es * row0 * P.C * P.h * P.r, 0,
                                 es * tail * P.C * P.h * P.r, st)) != cudaSuccess)
            return e;
    }
    if (fa.items == 0)  // nothing valid: every gradient, d_initial included, is zero
        return cudaMemsetAsync(A.dinit, 0, sizeof(float) * (size_t)P.b * P.h * P.p * P.r, st);
    TensorMaps maps;
    if ((e = encode_maps(P, A.xhat, A.bhat, A.rot, A.da, &maps)) != cudaSuccess) return e;
    int grid = fa.items < sm_count() ? fa.items : sm_count();
    if (!A.reuse_carries) {  // else the forward of the same problem left the carries in Hc / Dn
        if ((e = launch_tc_end(fa, maps, st)) != cudaSuccess) return e;
        if ((e = generic_carry_scan(P, A.initial, A.Hc, A.Dn, st)) != cudaSuccess) return e;
    }
    if (grid > kMaxBwdGrid) grid = kMaxBwdGrid;
    float* anchors = reinterpret_cast<float*>(scratch);
    float* drot2 = reinterpret_cast<float*>(scratch + bwd_anchor_bytes());
    if ((e = launch_tc_bwd(fa, A.E, anchors, drot2, A.dm2, A.dm1, A.dxhat, A.dbhat, A.dda, A.drot, maps, grid, st)) !=
        cudaSuccess)
        return e;
    if ((e = generic_cot_scan(P, A.E, A.Dn, A.dinit, st)) != cudaSuccess) return e;
    if ((e = encode_grad_maps(P, A.dxhat, A.dbhat, &maps)) != cudaSuccess) return e;
    return launch_tc_corr(fa, A.da, A.E, A.dxhat, A.dbhat, A.dda, maps, st);
}
