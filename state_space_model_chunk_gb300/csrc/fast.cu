// fast.cu -- host side of the tcgen05 path: eligibility, tensor-map encoding, dispatch.
#include <cuda.h>

#include <cstring>

#include "fast.h"
#include "fast_common.cuh"
#include "generic.h"
#include "prof.h"

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

size_t align256(size_t v) { return (v + 255) / 256 * 256; }

// The kernels' view of a problem: 64-token chunks, and each head's p state rows as p / 64 heads
// of 64 rows (MMParams::groups).
MMParams internal_params(const MMParams& P0) {
    MMParams P = P0;
    P.l = fastk::FL;
    P.nc = (P.s + fastk::FL - 1) / fastk::FL;
    P.heads = P0.h;
    P.groups = P0.p < 64 ? 1 : P0.p / 64;
    P.prow = P0.p < 64 ? P0.p : 64;  // below 64 rows: padded with zero rows
    P.h = P0.h * P.groups;
    P.p = 64;
    return P;
}

// p below 64: the caller's [b, h, prow, r] initial state into 64-row slots (rows past prow zero),
// and the kernels' 64-row d_initial back into the caller's layout.
__global__ void __launch_bounds__(256) k_pad_rows(const float* __restrict__ src, float* __restrict__ dst, int64_t bh,
                                                  int prow, int r) {
    const int64_t n = bh * 64 * r;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t u = i / ((int64_t)64 * r), rem = i - u * 64 * r;
        const int row = (int)(rem / r), col = (int)(rem - (int64_t)row * r);
        dst[i] = row < prow ? src[(u * prow + row) * r + col] : 0.f;
    }
}
__global__ void __launch_bounds__(256) k_unpad_rows(const float* __restrict__ src, float* __restrict__ dst, int64_t bh,
                                                    int prow, int r) {
    const int64_t n = bh * prow * r;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t u = i / ((int64_t)prow * r), rem = i - u * prow * r;
        dst[i] = src[u * 64 * r + rem];
    }
}
size_t padded_state_bytes(const MMParams& P) {  // P: the internal view
    return P.prow < P.p ? align256(sizeof(float) * (size_t)P.b * P.h * P.p * P.r) : 0;
}


// Workspace slices of a problem with several 64-row groups per head: the groups' own copies of
// the outputs that sum over state rows, added in group order once every group is done.
struct GroupSlices {
    size_t m2 = 0, m1 = 0, total_fwd = 0;                 // forward: m2 / m1 per group-head
    size_t db = 0, dda = 0, drot = 0, total_bwd = 0;      // backward: d_bhat, d_da, d_rot (+ drot2)
};

GroupSlices group_slices(const MMParams& P) {  // P: the internal view
    GroupSlices g;
    if (P.groups <= 1) return g;
    const size_t ntok = (size_t)P.b * P.s, G = (size_t)P.groups;
    g.m2 = 0;
    g.m1 = align256(sizeof(float) * (size_t)P.b * P.h * P.r * P.r);
    g.total_fwd = g.m1 + align256(sizeof(float) * (size_t)P.b * P.h * P.r);
    g.db = 0;
    g.dda = align256(2 * G * ntok * P.C * P.heads * P.r);
    g.drot = g.dda + align256(sizeof(float) * G * ntok * P.heads);
    // drot: the G slices of the rows-0-31 partials, then the G slices of the rows-32-63 ones
    g.total_bwd = g.drot + align256(sizeof(float) * 2 * G * ntok * P.heads * P.rw);
    return g;
}

// out[o][i] = sum over g = 0 .. G-1, in that order, of in[o][g][i] (fp32 sums).
__global__ void __launch_bounds__(256) k_group_sum_f32(const float* __restrict__ in, float* __restrict__ out,
                                                       int64_t outer, int G, int64_t inner) {
    const int64_t n = outer * inner;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t o = i / inner, e = i - o * inner;
        const float* src = in + o * G * inner + e;
        float acc = src[0];
        for (int g = 1; g < G; ++g) acc += src[(int64_t)g * inner];
        out[i] = acc;
    }
}

// The same over bf16 slices, eight elements per thread (inner a multiple of 8), rounded once.
__global__ void __launch_bounds__(256) k_group_sum_bf16(const uint4* __restrict__ in, uint4* __restrict__ out,
                                                        int G, int64_t inner8) {
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < inner8; i += (int64_t)gridDim.x * blockDim.x) {
        float acc[8];
        for (int g = 0; g < G; ++g) {
            const uint4 v = in[(int64_t)g * inner8 + i];
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float lo = __uint_as_float(w[j] << 16), hi = __uint_as_float(w[j] & 0xFFFF0000u);
                acc[2 * j] = g ? acc[2 * j] + lo : lo;
                acc[2 * j + 1] = g ? acc[2 * j + 1] + hi : hi;
            }
        }
        out[i] = make_uint4(tc::pack_bf16x2(acc[0], acc[1]), tc::pack_bf16x2(acc[2], acc[3]),
                            tc::pack_bf16x2(acc[4], acc[5]), tc::pack_bf16x2(acc[6], acc[7]));
    }
}

unsigned sum_blocks(int64_t n) {
    const int64_t cap = (int64_t)fastk::sm_count() * 8;
    const int64_t b = (n + 255) / 256;
    return (unsigned)(b < 1 ? 1 : (b > cap ? cap : b));
}

cudaError_t group_sum_f32(const float* in, float* out, int64_t outer, int G, int64_t inner, cudaStream_t st) {
    if (outer * inner == 0) return cudaSuccess;
    mm_prof_mark(KID_GROUP_SUM, 1, st);
    k_group_sum_f32<<<sum_blocks(outer * inner), 256, 0, st>>>(in, out, outer, G, inner);
    mm_prof_mark(KID_GROUP_SUM, 0, st);
    return cudaGetLastError();
}

cudaError_t group_sum_bf16(const void* in, void* out, int G, int64_t inner, cudaStream_t st) {
    if (inner == 0) return cudaSuccess;
    mm_prof_mark(KID_GROUP_SUM, 1, st);
    k_group_sum_bf16<<<sum_blocks(inner / 8), 256, 0, st>>>(static_cast<const uint4*>(in), static_cast<uint4*>(out), G,
                                                            inner / 8);
    mm_prof_mark(KID_GROUP_SUM, 0, st);
    return cudaGetLastError();
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
    {   // as x32, over d_xhat (the stores skip rows past prow)
        cuuint64_t dims[4] = {(cuuint64_t)P.prow, (cuuint64_t)P.h, (cuuint64_t)P.C, bs};
        cuuint64_t str[3] = {(cuuint64_t)P.prow * 2, (cuuint64_t)P.h * P.prow * 2, (cuuint64_t)P.C * P.h * P.prow * 2};
        cuuint32_t box[4] = {64, 1, (cuuint32_t)P.C, (cuuint32_t)corr_tps(P)};
        if ((e = encode(&maps->dx32, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, dx, dims, str, box,
                        CU_TENSOR_MAP_SWIZZLE_128B)) != cudaSuccess)
            return e;
    }
    {   // as b32, over d_bhat (a box's columns past r are skipped by the stores); with several row
        // groups, over their d_bhat slices, one after the other (rows group-major)
        cuuint64_t dims[4] = {(cuuint64_t)P.r, (cuuint64_t)P.heads, (cuuint64_t)P.C, bs * (cuuint64_t)P.groups};
        cuuint64_t str[3] = {(cuuint64_t)P.r * 2, (cuuint64_t)P.heads * P.r * 2, (cuuint64_t)P.C * P.heads * P.r * 2};
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
    {   // xhat as [b*s, C, h, prow] bf16 (h, prow: 64-row groups as heads); box = the C rows of one
        // (token, head), 64 wide: rows past prow (p below 64) read as zeros
        cuuint64_t dims[4] = {(cuuint64_t)P.prow, (cuuint64_t)P.h, (cuuint64_t)P.C, bs};
        cuuint64_t str[3] = {(cuuint64_t)P.prow * 2, (cuuint64_t)P.h * P.prow * 2, (cuuint64_t)P.C * P.h * P.prow * 2};
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
    {   // bhat as [b*s, C, heads, r] bf16; box = 64 columns (from column 64 a) of the C rows: columns
        // past r read as zeros, so an r below 128 leaves the tiles' tail zero
        cuuint64_t dims[4] = {(cuuint64_t)P.r, (cuuint64_t)P.heads, (cuuint64_t)P.C, bs};
        cuuint64_t str[3] = {(cuuint64_t)P.r * 2, (cuuint64_t)P.heads * P.r * 2, (cuuint64_t)P.C * P.heads * P.r * 2};
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
    if (P.rw > 0) {  // rot as [b*s, heads, rw] fp32; box = one (token, head)
        cuuint64_t dims[3] = {(cuuint64_t)P.rw, (cuuint64_t)P.heads, bs};
        cuuint64_t str[2] = {(cuuint64_t)P.rw * 4, (cuuint64_t)P.heads * P.rw * 4};
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
    } else {   // da as [b*s, heads] fp32; box = 4 heads of one token (16 bytes)
        cuuint64_t dims[2] = {(cuuint64_t)P.heads, bs};
        cuuint64_t str[1] = {(cuuint64_t)P.heads * 4};
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
    if (P.r < 16 || P.r > 128 || P.r % 16 || P.C < 1 || P.C > 8) return false;
    if (P.rot == ROT_HALF && P.r != 64 && P.r != 128) return false;
    // p: groups of 64 state rows, each run as a head of its own (grid rows and tensor-copy
    // coordinates of the groups stay within their 16- and 32-bit limits)
    // (below 64: the kernels run 64 rows, the rows past p zero; the caller's rows must stay 16-byte
    // multiples for the tensor copies)
    const bool small = P.p >= 8 && P.p < 64 && P.p % 8 == 0;
    if (!small && (P.p < 64 || P.p % 64 || P.p > 512)) return false;
    const int64_t groups = small ? 1 : P.p / 64;
    if ((int64_t)P.h * groups > 65535 || groups * P.b * P.s > ((int64_t)1 << 31) - 1) return false;
    if (P.b > MM_MAX_B) return false;  // (any s: the last chunk of a row may be partial)
    // rows of angles / quaternions are copied as 16-byte multiples, at most 128 floats
    if (P.rw % 4 || P.rw > 128) return false;
    if (!encode_fn()) return false;
    return true;
}

size_t fast_scratch_bytes(const MMParams& P, int backward) {
    const MMParams Pi = internal_params(P);
    const GroupSlices g = group_slices(Pi);
    if (!backward) return align256(fastk::fwd_partial_bytes(Pi)) + g.total_fwd + padded_state_bytes(Pi);
    const size_t a = fastk::bwd_anchor_bytes();  // a multiple of 256 bytes
    // (with row groups the d_rot partials live in the group slices); then the padded initial
    // state and d_initial for p below 64
    return a + (Pi.groups > 1 ? g.total_bwd : align256(fastk::bwd_drot2_bytes(P))) + 2 * padded_state_bytes(Pi);
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
    const GroupSlices gs = group_slices(P);
    char* gbase = scratch + align256(fwd_partial_bytes(P));
    if (P.groups > 1) {  // each group's moments into its own slice (zero where a group has no items)
        fa.m2 = reinterpret_cast<float*>(gbase + gs.m2);
        fa.m1 = reinterpret_cast<float*>(gbase + gs.m1);
        if ((e = cudaMemsetAsync(gbase, 0, gs.total_fwd, st)) != cudaSuccess) return e;
    }
    int grid = fa.items < sm_count() ? fa.items : sm_count();
    if (grid > kMaxFwdGrid) grid = kMaxFwdGrid;
    const float* init = A.initial;
    if (P.prow < P.p) {  // p below 64: the initial state in 64-row slots
        float* init64 = reinterpret_cast<float*>(gbase + gs.total_fwd);
        const int64_t bh = (int64_t)P.b * P.h;
        k_pad_rows<<<sum_blocks(bh * P.p * P.r), 256, 0, st>>>(A.initial, init64, bh, P.prow, P.r);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        init = init64;
    }
    if ((e = launch_tc_end(fa, maps, st)) != cudaSuccess) return e;
    if ((e = generic_carry_scan(P, init, A.Hc, A.Dn, st)) != cudaSuccess) return e;
    if ((e = launch_tc_fwd(fa, maps, grid, st)) != cudaSuccess || P.groups == 1) return e;
    // m2 / m1 of a head: its groups' moments, in group order
    const int64_t bh = (int64_t)P.b * P.heads;
    if ((e = group_sum_f32(fa.m2, A.m2, bh, P.groups, (int64_t)P.r * P.r, st)) != cudaSuccess) return e;
    return group_sum_f32(fa.m1, A.m1, bh, P.groups, P.r, st);
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
    const size_t bs = (size_t)P.b * P.s, es = 2;
    const size_t nx = bs * P.C * P.h * P.prow, nb = bs * P.C * P.heads * P.r, nda = bs * P.heads,
                 nrot = bs * P.heads * P.rw;
    if (fa.items == 0) {  // nothing valid: every gradient, d_initial included, is zero
        if ((e = cudaMemsetAsync(A.dxhat, 0, es * nx, st)) != cudaSuccess ||
            (e = cudaMemsetAsync(A.dbhat, 0, es * nb, st)) != cudaSuccess ||
            (e = cudaMemsetAsync(A.dda, 0, sizeof(float) * nda, st)) != cudaSuccess ||
            (P.rw && (e = cudaMemsetAsync(A.drot, 0, sizeof(float) * nrot, st)) != cudaSuccess))
            return e;
        return cudaMemsetAsync(A.dinit, 0, sizeof(float) * (size_t)P.b * P.h * P.prow * P.r, st);
    }
    // Where the kernels write d_bhat, d_da and d_rot: the outputs themselves (d_rot's second
    // partial in the workspace), or with several row groups one slice per group in the workspace,
    // added in group order at the end.
    const bool grouped = P.groups > 1;
    const GroupSlices gs = group_slices(P);
    char* gbase = scratch + bwd_anchor_bytes();
    void* db = grouped ? static_cast<void*>(gbase + gs.db) : A.dbhat;
    float* dda = grouped ? reinterpret_cast<float*>(gbase + gs.dda) : A.dda;
    float* drot = grouped ? reinterpret_cast<float*>(gbase + gs.drot) : A.drot;
    float* drot2 = grouped ? drot + (size_t)P.groups * nrot : reinterpret_cast<float*>(gbase);
    const int G = P.groups;
    // d_da and d_rot start from zero: the kernels write them for valid positions only (d_rot as
    // two partial sums that a second pass adds; d_da then gets the correction added).  d_xhat /
    // d_bhat at positions at or past valid_len are exactly zero; every position before is written.
    if ((e = cudaMemsetAsync(dda, 0, sizeof(float) * nda * G, st)) != cudaSuccess) return e;
    if (P.rw && (e = cudaMemsetAsync(drot, 0, sizeof(float) * nrot * (grouped ? 2 * G : 1), st)) != cudaSuccess)
        return e;
    for (int bb = 0; bb < P.b; ++bb) {
        const size_t v = (size_t)P.valid[bb], tail = (size_t)P.s - v;
        if (!tail) continue;
        const size_t row0 = (size_t)bb * P.s + v;
        if ((e = cudaMemsetAsync(static_cast<char*>(A.dxhat) + es * row0 * P.C * P.h * P.prow, 0,
                                 es * tail * P.C * P.h * P.prow, st)) != cudaSuccess)
            return e;
        for (int g = 0; g < G; ++g)
            if ((e = cudaMemsetAsync(static_cast<char*>(db) + es * ((size_t)g * nb + row0 * P.C * P.heads * P.r), 0,
                                     es * tail * P.C * P.heads * P.r, st)) != cudaSuccess)
                return e;
    }
    TensorMaps maps;
    if ((e = encode_maps(P, A.xhat, A.bhat, A.rot, A.da, &maps)) != cudaSuccess) return e;
    int grid = fa.items < sm_count() ? fa.items : sm_count();
    // p below 64: the initial state and d_initial in 64-row slots after the other scratch
    char* pbase = scratch + bwd_anchor_bytes() + (grouped ? gs.total_bwd : align256(bwd_drot2_bytes(P0)));
    float* init64 = reinterpret_cast<float*>(pbase);
    float* dinit64 = reinterpret_cast<float*>(pbase + padded_state_bytes(P));
    const bool padded = P.prow < P.p;
    const int64_t bh = (int64_t)P.b * P.h;
    if (!A.reuse_carries) {  // else the forward of the same problem left the carries in Hc / Dn
        const float* init = A.initial;
        if (padded) {
            k_pad_rows<<<sum_blocks(bh * P.p * P.r), 256, 0, st>>>(A.initial, init64, bh, P.prow, P.r);
            if ((e = cudaGetLastError()) != cudaSuccess) return e;
            init = init64;
        }
        if ((e = launch_tc_end(fa, maps, st)) != cudaSuccess) return e;
        if ((e = generic_carry_scan(P, init, A.Hc, A.Dn, st)) != cudaSuccess) return e;
    }
    if (grid > kMaxBwdGrid) grid = kMaxBwdGrid;
    float* anchors = reinterpret_cast<float*>(scratch);
    if ((e = launch_tc_bwd(fa, A.E, anchors, drot2, A.dm2, A.dm1, A.dxhat, db, dda, drot, A.rot, maps, grid, st)) !=
        cudaSuccess)
        return e;
    if ((e = generic_cot_scan(P, A.E, A.Dn, padded ? dinit64 : A.dinit, st)) != cudaSuccess) return e;
    if (padded) {  // d_initial back into the caller's rows
        k_unpad_rows<<<sum_blocks(bh * P.prow * P.r), 256, 0, st>>>(dinit64, A.dinit, bh, P.prow, P.r);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    if ((e = encode_grad_maps(P, A.dxhat, db, &maps)) != cudaSuccess) return e;
    if ((e = launch_tc_corr(fa, A.da, A.E, A.dxhat, db, dda, maps, st)) != cudaSuccess || !grouped) return e;
    // a head's d_bhat, d_da and d_rot: its groups' slices in group order (d_rot: the G rows-0-31
    // partials, then the G rows-32-63 ones)
    if ((e = group_sum_bf16(db, A.dbhat, G, (int64_t)nb, st)) != cudaSuccess) return e;
    if ((e = group_sum_f32(dda, A.dda, 1, G, (int64_t)nda, st)) != cudaSuccess) return e;
    if (P.rw && (e = group_sum_f32(drot, A.drot, 1, 2 * G, (int64_t)nrot, st)) != cudaSuccess) return e;
    return launch_drot_finish(P, A.drot, nullptr, A.rot, st);  // quaternions: the factor Q / |Q|^2
}
