// fast_common.cuh -- pieces shared by the tensor-core kernels: launch arguments, the work-item
// enumeration (pairs of 64-token chunks of one (batch row, head)), the per-thread column
// groups of a 128-column row, and the register-level de-rotation / its transpose.
#pragma once
#include <cuda.h>

#include "common.cuh"
#include "tc.cuh"

namespace fastk {

constexpr int FL = 64;   // internal chunk length of the tensor-core path
constexpr int NCW = 8;   // compute warps (two threads per 128-column row)

struct FastArgs {
    MMParams P;     // internal chunking: l = 64, nc = s / 64
    int layoutB;    // 1: half-split rotation with r = 64 (partner columns 32 apart)
    int items;      // work items (chunk pairs) of the whole problem
    float* Hc;      // [b,h,nc,p,r] chunk carries / chunk-end states (h, p: the 64-row groups as heads)
    float* Dn;      // [b,h,nc] chunk decays
    float* m2;
    float* m1;
    const float* da;  // [b,s,h] (read with plain loads when h is not a multiple of 4)
    float* m2p;     // forward: per-CTA partial moments of (b,h) shared with other CTAs, 2 slots per CTA
                    // of r*r (m2) + r (m1) floats, summed in CTA order by the reduce kernel
    int* err;       // device error word (0 = fine)
    int test_wait_timeout;  // chunk-end kernel: one wait that nothing completes (failure-path test)
};

struct TensorMaps {
    CUtensorMap x, b, rot, da, da64;  // da: 4 heads x 1 token; da64: 4 heads x 64 tokens
    CUtensorMap x8, b8;               // xhat / bhat rows of 8 consecutive tokens
    CUtensorMap x32, b32;             // ... and of corr_tps(P) tokens (the correction kernel's stages)
    CUtensorMap dx32, db32;           // d_xhat / d_bhat rows of corr_tps(P) tokens (backward only)
};

constexpr int kMaxBwdGrid = 160;  // CTAs of the backward kernels (anchor slots in the workspace)
constexpr int kMaxFwdGrid = 160;  // CTAs of the forward kernel (partial-moment slots in the workspace)

__host__ __device__ inline int pairs_of(const MMParams& P, int bb) { return (mm_processed(P, bb) + 1) / 2; }

__host__ inline int count_items(const MMParams& P) {
    int n = 0;
    for (int bb = 0; bb < P.b; ++bb) n += P.h * pairs_of(P, bb);
    return n;
}

struct Item {
    int bb, hh, k;   // batch row, head, pair index (chunks 2k and 2k+1)
    int hd, grp;     // the caller's head and the 64-row group of hh (MMParams::groups)
    int proc;        // processed chunks of the row
    int T[2];        // valid tokens of both chunks (T[0] >= T[1])
    bool exists[2];  // chunk inside the sequence
    bool seg_first, seg_last;  // first / last item of this CTA's run on (bb, hh)
};

__device__ inline void locate(const FastArgs& A, int item, int& bb, int& hh, int& k) {
    const MMParams& P = A.P;
    int base = 0;
    for (bb = 0; bb < P.b - 1; ++bb) {
        int cnt = P.h * pairs_of(P, bb);
        if (item < base + cnt) break;
        base += cnt;
    }
    const int np = pairs_of(P, bb);
    const int rem = item - base;
    hh = rem / np;
    k = rem - hh * np;
}

__device__ inline int item_begin(const FastArgs& A, int cta) {
    return (int)(((int64_t)cta * A.items) / gridDim.x);
}
// The same for a kernel whose grid is not the one that walked the items.
__host__ __device__ inline int item_begin_of(int items, int grid, int cta) {
    return (int)(((int64_t)cta * items) / grid);
}

__device__ inline Item decode_item(const FastArgs& A, int item) {
    const MMParams& P = A.P;
    Item I;
    locate(A, item, I.bb, I.hh, I.k);
    I.hd = I.hh / P.groups;
    I.grp = I.hh - I.hd * P.groups;
    I.proc = mm_processed(P, I.bb);
    for (int ch = 0; ch < 2; ++ch) {
        const int n = 2 * I.k + ch;
        I.exists[ch] = n < P.nc;
        I.T[ch] = n < I.proc ? mm_chunk_rows(P, I.bb, n) : 0;
    }
    const int it0 = item_begin(A, blockIdx.x), it1 = item_begin(A, blockIdx.x + 1);
    I.seg_first = true;
    I.seg_last = true;
    if (item > it0) {
        int b2, h2, k2;
        locate(A, item - 1, b2, h2, k2);
        I.seg_first = !(b2 == I.bb && h2 == I.hh);
    }
    if (item + 1 < it1) {
        int b2, h2, k2;
        locate(A, item + 1, b2, h2, k2);
        I.seg_last = !(b2 == I.bb && h2 == I.hh);
    }
    return I;
}

struct TokenInfo {
    bool seg_first, seg_last;
};

// Flat walk over the tokens of a CTA's items (the MMA issuer's view).
struct TokenWalk {
    const FastArgs& A;
    int it, it1, t;
    Item I;
    __device__ TokenWalk(const FastArgs& a, int i0, int i1) : A(a), it(i0), it1(i1), t(0) {
        if (it < it1) I = decode_item(A, it);
    }
    __device__ uint32_t total_tokens() const {
        uint32_t n = 0;
        for (int i = it; i < it1; ++i) n += (uint32_t)decode_item(A, i).T[0];
        return n;
    }
    __device__ TokenInfo next() {
        while (t >= I.T[0] && it + 1 < it1) {
            ++it;
            t = 0;
            I = decode_item(A, it);
        }
        TokenInfo ti{I.seg_first && t == 0, I.seg_last && t == I.T[0] - 1};
        ++t;
        return ti;
    }
};

// da comes by tensor copies of 4-head groups when a row of da ([b*s, h] fp32) is a multiple of 16
// bytes long, else by plain loads of the one head into the same shared-memory positions.
__host__ __device__ inline bool da_by_tma(const MMParams& P) { return (P.heads & 3) == 0; }

// Tokens per stage of the correction kernel: their (token, channel) rows fill at most the 128
// lanes of one tensor-core tile.
__host__ __device__ inline int corr_tps(const MMParams& P) { return P.C <= 4 ? 32 : 16; }

// Transaction bytes of one chunk's share of a stage: C rows of xhat (64 bf16), C rows of each
// 64-wide half of bhat, one token's rotation parameters and one 16-byte group of da.
__host__ __device__ inline uint32_t stage_bytes(const FastArgs& A) {
    const MMParams& P = A.P;
    return 128u * P.C + (uint32_t)((P.r + 63) / 64) * 128u * P.C + 4u * P.rw + (da_by_tma(P) ? 16u : 0u);
}

// The four 16-column groups of a 128-column row that one thread owns.  Rotation partners
// always fall in the same thread: pairs (2i, 2i+1); half-split pairs (i, i + 64) for r = 128
// (layout A) or (i, i + 32) for r = 64 (layout B); quaternion 4-blocks.
__device__ inline void col_groups(int layoutB, int half, int (&G)[4]) {
    if (!layoutB) {
        G[0] = 2 * half; G[1] = 2 * half + 1; G[2] = 4 + 2 * half; G[3] = 5 + 2 * half;
    } else {
        G[0] = half; G[1] = 2 + half; G[2] = 4 + 2 * half; G[3] = 5 + 2 * half;
    }
}

__device__ __forceinline__ void named_barrier_sync(int id, int count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

__device__ __forceinline__ void hamilton(float qw, float qx, float qy, float qz, float vw, float vx, float vy,
                                         float vz, float& ow, float& ox, float& oy, float& oz) {
    ow = qw * vw - qx * vx - qy * vy - qz * vz;
    ox = qw * vx + qx * vw + qy * vz - qz * vy;
    oy = qw * vy - qx * vz + qy * vw + qz * vx;
    oz = qw * vz + qx * vy - qy * vx + qz * vw;
}

// Packed fp32x2 arithmetic (sm_100 and later): one instruction for two values, each rounded
// exactly as the scalar fmaf / product it replaces, so using it changes no result.
// (d0, d1) <- (a0, a1) * (b0, b1) + (c0, c1)
__device__ __forceinline__ void ffma2(float& d0, float& d1, float a0, float a1, float b0, float b1, float c0, float c1) {
    const float2 r = __ffma2_rn(make_float2(a0, a1), make_float2(b0, b1), make_float2(c0, c1));
    d0 = r.x;
    d1 = r.y;
}
// (d0, d1) <- (a0, a1) * (b0, b1)
__device__ __forceinline__ void fmul2(float& d0, float& d1, float a0, float a1, float b0, float b1) {
    const float2 r = __fmul2_rn(make_float2(a0, a1), make_float2(b0, b1));
    d0 = r.x;
    d1 = r.y;
}

__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// 16 columns (group gcol of 16) of row m of a bf16 [128 x 128] swizzled tile, from floats.
__device__ __forceinline__ void write_tile16(unsigned char* tile, int m, int gcol, const float (&v)[16], bool zero) {
    const uint32_t hv = gcol >> 2, j0 = 2 * (gcol & 3);
#pragma unroll
    for (int hj = 0; hj < 2; ++hj) {
        uint4 w = make_uint4(0, 0, 0, 0);
        if (!zero) {
            w.x = tc::pack_bf16x2(v[8 * hj + 0], v[8 * hj + 1]);
            w.y = tc::pack_bf16x2(v[8 * hj + 2], v[8 * hj + 3]);
            w.z = tc::pack_bf16x2(v[8 * hj + 4], v[8 * hj + 5]);
            w.w = tc::pack_bf16x2(v[8 * hj + 6], v[8 * hj + 7]);
        }
        *reinterpret_cast<uint4*>(tile + tc::sw128_chunk(128, hv, m, j0 + hj)) = w;
    }
}

// Slots of a 32-column pass: rotation partners stay inside (half-split, r = 64: slots 0/1).
template <int LAYB>
__device__ __forceinline__ int slot_a(int pass) { return LAYB ? 2 * pass : pass; }
template <int LAYB>
__device__ __forceinline__ int slot_b(int pass) { return LAYB ? 2 * pass + 1 : pass + 2; }

// Whether the 16-column group gcol holds rotated columns (pairs, x halves or 4-blocks whose
// angle / quaternion index lies below the rotated width); the others rotate by the identity.
template <int ROTK>
__device__ __forceinline__ bool group_rotated(const MMParams& P, int gcol) {
    if (ROTK == ROT_PAIRWISE) return 8 * gcol < P.na;
    if (ROTK == ROT_HALF) return 16 * gcol < P.na;
    if (ROTK == ROT_QUAT) return 4 * gcol < P.J;
    return false;
}

// host helpers
cudaError_t encode_maps(const MMParams& P, const void* xhat, const void* bhat, const float* rot, const float* da,
                        TensorMaps* maps);
int sm_count();
cudaError_t launch_tc_fwd(const FastArgs& args, const TensorMaps& maps, int grid, cudaStream_t st);
cudaError_t launch_tc_end(const FastArgs& fa, const TensorMaps& maps, cudaStream_t st);
// Tensor maps over the d_xhat / d_bhat outputs, same geometry as x32 / b32.
cudaError_t encode_grad_maps(const MMParams& P, const void* dx, const void* db, TensorMaps* maps);
cudaError_t launch_tc_corr(const FastArgs& fa, const float* da, const float* E, void* dx, void* db, float* dda,
                           const TensorMaps& maps, cudaStream_t st);
size_t bwd_anchor_bytes();
size_t bwd_drot2_bytes(const MMParams& P);  // the backward's second d_rot partial, [b,s,h,rw] fp32
size_t fwd_partial_bytes(const MMParams& P);  // internal chunking (nc = s / 64)
// rot: the cumulative rotation (quaternions: d_rot is finished with each block's Q / |Q|^2)
cudaError_t launch_tc_bwd(const FastArgs& fa, float* E, float* anchors, float* drot2, const float* dm2, const float* dm1,
                          void* dx, void* db, float* dda, float* drot, const float* rot, const TensorMaps& maps, int grid,
                          cudaStream_t st);
// d_rot from the backward's partial sums: drot += drot2 (drot2 may be null), then for quaternions
// the factor Q / |Q|^2 of each block; positions past valid_len stay as they are
cudaError_t launch_drot_finish(const MMParams& P, float* drot, const float* drot2, const float* rot, cudaStream_t st);

}  // namespace fastk
