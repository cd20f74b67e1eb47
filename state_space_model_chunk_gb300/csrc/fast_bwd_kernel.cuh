// fast_bwd_kernel.cuh -- tcgen05 / TMA recompute backward of the state-moments operator (bf16 operands,
// 64 state rows per head -- larger p as 64-row groups run as heads --, r up to 128, C <= 8).
//
// Work item = a pair of 64-token chunks of one (batch row, head); the two chunks share the 128
// TMEM lanes (row m = (chunk, p)) as in the forward.  This kernel is the chunk's own backward with
// zero incoming carry cotangent ("backward.rs", module header "Gradient math", with the d_h+
// term split off; fast_corr.cu adds it once the cotangent scan has run):
//   phase A  forward sweep from the chunk carry, one 8-token span at a time: S <- D_k S +
//            sum_j L[end, j] W_j with the sum as one K = 128 tensor-core product (xhat rows scaled
//            in place by L); the state after every 8th token is kept as an fp32 anchor in this
//            CTA's workspace slot (7 anchors; the chunk carry is anchor 0), column-quad-major.
//   phase B  8-token spans in reverse.  For token t of a span starting at s0 the state is
//            rebuilt exactly as  h_t = exp(a_t - a_anchor) A + sum_{s0<=j<=t} L[t,j] W_j : one
//            prefix product with one K = 16 step per span token j <= t (A rows = xhat rows scaled
//            by L[t,j] = exp(a_t - a_j)), plus the anchor term read from TMEM.  Then c = derot(h)
//            as bf16 pairs into TMEM, d_c = c (D + D^T) + 1 d_m1^T on tcgen05 with A = that c
//            tile (K = r, and one K = 16 step for d_m1), d_rot from (c, d_c) by warp transpose
//            reductions over p, G = derot^T(d_c), the cotangent recurrence g_t = G_t + e_{t+1}
//            g_{t+1} in registers, d_da_{t+1} = e_{t+1} <g_{t+1}, h_t>, and d_xhat = g bhat^T,
//            d_bhat = g^T xhat as N = 16 MMAs.  After the chunk: e_n = e_0 g_0.
//            The span is software-pipelined: while the CUDA cores finish the cotangent work of
//            token t, the tensor cores already run d_c of token t-1 and the prefix of t-2.  The
//            span's token slots are released one by one (token s0 + j's d_xhat / d_bhat product
//            is the last reader of slot j), so the next span's high slots load early.
//
// Warp roles: 0-7 compute (two threads per row, 64 columns each, handled as two 32-column
// passes whose rotation partners stay inside the pass), 8 TMA (all 32 lanes issue copies), 9 MMA.
// d_rot and d_da are summed over each warp's 32 rows with warp transpose-reductions; the two
// warps of a chunk's 64 rows are then combined in a fixed order (d_da through shared memory at
// the end of the item, d_rot by k_drot_finish after the kernel).  Every wait is bounded; a
// timeout sets the workspace error word and the CTA winds down.
#pragma once
#include <cuda.h>

#include "common.cuh"
#include "fast.h"
#include "fast_common.cuh"
#include "prof.h"
#include "tc.cuh"

namespace fastbwd {

using namespace fastk;

constexpr int NTHR = 320;
constexpr int WARP_TMA = 8, WARP_MMA = 9;
constexpr int SPAN = 8;        // tokens per anchor span
constexpr int NANCHOR = 7;     // anchors per 64-token chunk kept in the workspace (anchor 0 = carry)

// shared memory map (bytes from a 1024-aligned base)
constexpr uint32_t OFF_G = 0;                    // g tile [128 rows (ch,p)][128 r] bf16, 32 KB
constexpr uint32_t OFF_DS = 32768;               // D + D^T    [128 r2][128 r1] bf16
constexpr uint32_t OFF_SX = 65536;               // span xhat tiles, 8 x [16 rows (8ch+c)][128 (ch,p)]
constexpr uint32_t OFF_SB = 98304;               // span bhat tiles, 8 x [16 rows (8ch+c)][128 r]
constexpr uint32_t OFF_PA = 131072;              // prefix A tiles, 8 x [16 rows (8ch+c)][128 (ch,p)]
constexpr uint32_t OFF_ROT = 163840;             // span rotation rows, 8 tokens x 2 chunks x 512 B
constexpr uint32_t OFF_IDA = 172032;             // item da: 2 chunks x 64 tokens x 4 heads fp32
constexpr uint32_t OFF_ACUM = 174080;            // cumulative da, 2 chunks x 64 fp32
constexpr uint32_t OFF_COEF = 174592;            // span cos|sin: 8 tokens x 2 chunks x 128 fp32
constexpr uint32_t OFF_LT = 182784;              // span decay matrix L: 2 chunks x 8 x 8 fp32
constexpr uint32_t OFF_M1T = 184320;             // d_m1 as a K = 16 MMA operand: rows hi | lo (bf16) | 0
constexpr uint32_t OFF_PTR = 188416;             // per compute thread: 3 output row pointers of the item
constexpr uint32_t OFF_DDA = 194560;             // d_da partials of the item: [2 chunks][64 tokens][4 warps]
constexpr uint32_t OFF_CTL = 196608;
constexpr uint32_t SMEM_BYTES = OFF_CTL + 512 + 1024;
static_assert(OFF_SX % 1024 == 0 && OFF_SB % 1024 == 0 && OFF_PA % 1024 == 0 && OFF_M1T % 1024 == 0, "tiles");
static_assert(OFF_ROT % 128 == 0 && OFF_IDA % 128 == 0 && OFF_CTL % 8 == 0, "tensor-copy slots");
static_assert(OFF_PTR + 256 * 3 * 8 <= OFF_DDA && OFF_DDA + 2 * 64 * 4 * 4 <= OFF_CTL, "pointer table, d_da partials");
static_assert(SMEM_BYTES <= 232448, "shared memory");

struct Ctl {
    uint64_t itemfull, itemdone;
    uint64_t afull[2], ascaled[2], aempty[2];  // forward-sweep span buffers
    uint64_t wfull[2], wfree[2];
    uint64_t spanfull;
    uint64_t slotfree[8];  // span slot j (xhat, bhat, rotation rows of one token) read for the last time
    uint64_t pafull, pafree, pfull, pfree;
    uint64_t cfull, cfree, dcfull, dcfree;
    uint64_t gfull, gfree, dxfull, dxfree;
    uint64_t fin;
    uint32_t tbase;
    int abort;
    int loaded_b, loaded_h;
    float* dda_row[2];  // d_da of the item's two chunks at token 0 (the row stride is the head count)
    int tvalid[2];      // valid tokens of the item's two chunks (RAG)
};
static_assert(sizeof(Ctl) <= 512, "control block");

// tensor memory columns; CA holds the c tile as bf16 pairs (row = lane), the A operand of the
// d_c product, so the c tile needs no shared memory; ONE is a K = 16 A operand whose first two
// columns are 1, so that one more step of that product adds d_m1 (hi + lo) to every row
constexpr uint32_t TM_P = 0, TM_DC = 128, TM_AN = 256, TM_DX = 384, TM_DB = 400, TM_CA = 416, TM_ONE = 480,
                   TM_COLS = 512;

// Position of state element (row m, columns col .. col+3) in an anchor of the workspace: 16-byte
// pieces ordered column-quad-major, so that the 32 rows of a warp touch 512 contiguous bytes
// per access (each thread owns one row).
__device__ __forceinline__ int64_t anchor_off(int m, int col) { return ((int64_t)(col >> 2) * 128 + m) * 4; }

// c-tile row of one 16-column group in tensor memory: 16 bf16, two per 32-bit column
__device__ __forceinline__ void ca_store16(uint32_t taddr, const float (&v)[16], bool zero) {
    uint32_t w[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) w[j] = zero ? 0u : tc::pack_bf16x2(v[2 * j], v[2 * j + 1]);
    tc::tmem_st8u(taddr, w);
}
__device__ __forceinline__ void ca_load16(uint32_t taddr, float (&v)[16]) {
    uint32_t w[8];
    tc::tmem_ld8u(taddr, w);
    tc::tmem_wait_ld();
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        v[2 * j] = bf16lo(w[j]);
        v[2 * j + 1] = bf16hi(w[j]);
    }
}

// eight bf16 values (one 16-byte piece of a tile) times L, rounded back to bf16
__device__ __forceinline__ uint4 scale_bf16x8(const uint4 v, float L) {
    float f[8];
    fmul2(f[0], f[1], L, L, bf16lo(v.x), bf16hi(v.x));
    fmul2(f[2], f[3], L, L, bf16lo(v.y), bf16hi(v.y));
    fmul2(f[4], f[5], L, L, bf16lo(v.z), bf16hi(v.z));
    fmul2(f[6], f[7], L, L, bf16lo(v.w), bf16hi(v.w));
    return make_uint4(tc::pack_bf16x2(f[0], f[1]), tc::pack_bf16x2(f[2], f[3]), tc::pack_bf16x2(f[4], f[5]),
                      tc::pack_bf16x2(f[6], f[7]));
}

struct BwdArgs {
    FastArgs F;         // problem, items, Hc (carries), Dn, err
    float* E;           // [b,h,nc,p,r]: e_n of every chunk
    float* anchors;     // [grid][7] fp32 anchor slots of 128 x 128, laid out by anchor_off
    const float* dm2;   // [b,h,r,r]
    const float* dm1;   // [b,h,r]
    __nv_bfloat16* dx;  // d_xhat
    __nv_bfloat16* db;  // d_bhat
    float* dda;         // d_da (zeroed by the host; added into)
    float* drot;        // d_rot (zeroed by the host): partial sums over rows 0-31 of each chunk
    float* drot2;       // [b,s,h,rw] workspace: partial sums over rows 32-63
    // elements between the slices of consecutive 64-row groups (MMParams::groups) in db, dda,
    // drot and drot2; 0 with one group
    int64_t db_slice, dda_slice, drot_slice;
};

__device__ __forceinline__ void fail(Ctl* ctl, int* err, int code) {
    ctl->abort = 1;
    atomicExch(err, code);
}

// Sum of 16 per-lane values across the warp, transposed: on return v[0] of lane L holds the sum
// over all lanes of the original v[L & 15].
__device__ __forceinline__ void transpose_reduce16(float (&v)[16], int lane) {
#pragma unroll
    for (int off = 8; off >= 1; off >>= 1) {
        const bool upper = (lane & off) != 0;
#pragma unroll
        for (int i = 0; i < off; ++i) {
            const float send = upper ? v[i] : v[i + off];
            const float keep = upper ? v[i + off] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
        }
    }
    v[0] += __shfl_xor_sync(0xffffffffu, v[0], 16);
}

// The same for 8 values: on return v[0] of lane L holds the sum over all lanes of v[L & 7].
__device__ __forceinline__ void transpose_reduce8(float (&v)[8], int lane) {
#pragma unroll
    for (int off = 4; off >= 1; off >>= 1) {
        const bool upper = (lane & off) != 0;
#pragma unroll
        for (int i = 0; i < off; ++i) {
            const float send = upper ? v[i] : v[i + off];
            const float keep = upper ? v[i + off] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
        }
    }
    v[0] += __shfl_xor_sync(0xffffffffu, v[0], 8);
    v[0] += __shfl_xor_sync(0xffffffffu, v[0], 16);
}

// (out_a, out_b) = rotation of the two slots of a pass: de-rotation R(-theta) / Q (x) . (TR =
// false) or its transpose (TR = true).  cf: cos at [0,64), sin at [64,128) of this token and
// chunk's angles; qt: its raw quaternions.  ka / kb: first column of slot a / b.
template <int ROTK, int LAYB, bool TR>
__device__ __forceinline__ void rot_pass(const MMParams& P, int pass, int ka, int kb, bool act_a, bool act_b,
                                         float (&a)[16], float (&b)[16], const float* cf, const float* qt) {
    // cf holds cos / sin for all 64 angle slots; slots at or past the rotated width hold (1, 0)
    if (ROTK == ROT_PAIRWISE) {
#pragma unroll
        for (int s = 0; s < 2; ++s) {
            if (!(s ? act_b : act_a)) continue;
            float(&v)[16] = s ? b : a;
            const int i0 = (s ? kb : ka) >> 1;  // 8 consecutive angles
            float cs[8], sn[8];
            *reinterpret_cast<float4*>(&cs[0]) = *reinterpret_cast<const float4*>(cf + i0);
            *reinterpret_cast<float4*>(&cs[4]) = *reinterpret_cast<const float4*>(cf + i0 + 4);
            *reinterpret_cast<float4*>(&sn[0]) = *reinterpret_cast<const float4*>(cf + 64 + i0);
            *reinterpret_cast<float4*>(&sn[4]) = *reinterpret_cast<const float4*>(cf + 64 + i0 + 4);
#pragma unroll
            for (int e = 0; e < 16; e += 2) {
                const float c_ = cs[e / 2], s_ = TR ? -sn[e / 2] : sn[e / 2];
                const float x = v[e], y = v[e + 1];
                v[e] = fmaf(c_, x, s_ * y);
                v[e + 1] = fmaf(c_, y, -s_ * x);
            }
        }
    } else if (ROTK == ROT_HALF) {
        if ((LAYB && pass == 1) || !act_a) return;  // padding columns of r = 64 / identity
#pragma unroll
        for (int e4 = 0; e4 < 16; e4 += 4) {
            const float4 c4 = *reinterpret_cast<const float4*>(cf + ka + e4);
            const float4 s4 = *reinterpret_cast<const float4*>(cf + 64 + ka + e4);
            const float cs[4] = {c4.x, c4.y, c4.z, c4.w}, sn[4] = {s4.x, s4.y, s4.z, s4.w};
#pragma unroll
            for (int j = 0; j < 4; j += 2) {
                const int e = e4 + j;
                const float s0 = TR ? -sn[j] : sn[j], s1 = TR ? -sn[j + 1] : sn[j + 1];
                const float x0 = a[e], x1 = a[e + 1], y0 = b[e], y1 = b[e + 1];
                float u0, u1, w0, w1;
                fmul2(u0, u1, s0, s1, y0, y1);    // s y
                fmul2(w0, w1, -s0, -s1, x0, x1);  // -s x
                ffma2(a[e], a[e + 1], cs[j], cs[j + 1], x0, x1, u0, u1);
                ffma2(b[e], b[e + 1], cs[j], cs[j + 1], y0, y1, w0, w1);
            }
        }
    } else if (ROTK == ROT_QUAT) {
#pragma unroll
        for (int s = 0; s < 2; ++s) {
            if (!(s ? act_b : act_a)) continue;
            float(&v)[16] = s ? b : a;
            const int k0 = s ? kb : ka;
#pragma unroll
            for (int e = 0; e < 16; e += 4) {
                const int blk = (k0 + e) >> 2;
                if (blk < P.J) {
                    const float* Q = qt + 4 * blk;
                    const float qx = TR ? -Q[1] : Q[1], qy = TR ? -Q[2] : Q[2], qz = TR ? -Q[3] : Q[3];
                    hamilton(Q[0], qx, qy, qz, v[e], v[e + 1], v[e + 2], v[e + 3], v[e], v[e + 1], v[e + 2], v[e + 3]);
                }
            }
        }
    }
}

// Parities of the barriers a thread waits on, one bit each, and one-bit "used before" flags,
// all in one register.
struct Par {
    uint32_t b = 0;
    __device__ __forceinline__ uint32_t next(uint32_t i) {
        const uint32_t p = (b >> i) & 1u;
        b ^= 1u << i;
        return p;
    }
    __device__ __forceinline__ bool once(uint32_t i) {  // false the first time, true afterwards
        const bool was = (b >> i) & 1u;
        b |= 1u << i;
        return was;
    }
};
// bit positions
enum : uint32_t {
    B_W = 4,                          // 2 W buffers
    B_ITEM = 6, B_SPAN, B_PA, B_P, B_C, B_DC, B_G, B_DX, B_ITEMDONE,
    U_PRE = 24, U_DC, U_DX, U_PA, U_C, U_G, U_SPAN
};
// RAG: the general-shape variant, for a sequence length that is not a multiple of 64 (a row's last
// chunk ends inside it: the second chunk of a pair stores its per-token gradient rows only up to
// its valid tokens, its steps running on with the first chunk's past the row's end) and for fewer
// than 64 state rows per head (the d_xhat rows past prow, zero padding, are not stored)
template <int ROTK, int LAYB, int CS, bool RAG>
__global__ void __launch_bounds__(NTHR, 1)
    tc_bwd_kernel(const __grid_constant__ BwdArgs B, const __grid_constant__ CUtensorMap tmx,
                  const __grid_constant__ CUtensorMap tmb, const __grid_constant__ CUtensorMap tmr,
                  const __grid_constant__ CUtensorMap tmd) {
    extern __shared__ unsigned char smraw[];
    unsigned char* sm = smraw + ((1024u - (tc::smem_u32(smraw) & 1023u)) & 1023u);
    Ctl* ctl = reinterpret_cast<Ctl*>(sm + OFF_CTL);
    const FastArgs& A = B.F;
    const MMParams& P = A.P;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int R = P.r, C = P.C;
    const int it0 = item_begin(A, blockIdx.x), it1 = item_begin(A, blockIdx.x + 1);

    // ---- set-up: zero the operand tiles whose padding rows/halves must read as zero
    for (uint32_t i = tid; i < (OFF_ROT - OFF_G) / 16; i += NTHR)
        reinterpret_cast<uint4*>(sm + OFF_G)[i] = make_uint4(0, 0, 0, 0);
    for (uint32_t i = tid; i < (OFF_CTL - OFF_ROT) / 4; i += NTHR) reinterpret_cast<float*>(sm + OFF_ROT)[i] = 0.f;
    if (tid == 0) {
        tc::mbar_init(&ctl->itemfull, 1);
        tc::mbar_init(&ctl->itemdone, NCW);
        for (int i = 0; i < 2; ++i) {
            tc::mbar_init(&ctl->afull[i], 1);
            tc::mbar_init(&ctl->ascaled[i], NCW);
            tc::mbar_init(&ctl->aempty[i], 1 + NCW);
            tc::mbar_init(&ctl->wfull[i], 1);
            tc::mbar_init(&ctl->wfree[i], NCW);
        }
        tc::mbar_init(&ctl->spanfull, 1);
        for (int j = 0; j < SPAN; ++j) tc::mbar_init(&ctl->slotfree[j], 1);
        tc::mbar_init(&ctl->pafull, NCW);
        tc::mbar_init(&ctl->pafree, 1);
        tc::mbar_init(&ctl->pfull, 1);
        tc::mbar_init(&ctl->pfree, NCW);
        tc::mbar_init(&ctl->cfull, NCW);
        tc::mbar_init(&ctl->cfree, 1);
        tc::mbar_init(&ctl->dcfull, 1);
        tc::mbar_init(&ctl->dcfree, NCW);
        tc::mbar_init(&ctl->gfull, NCW);
        tc::mbar_init(&ctl->gfree, 1);
        tc::mbar_init(&ctl->dxfull, 1);
        tc::mbar_init(&ctl->dxfree, NCW);
        tc::mbar_init(&ctl->fin, 1);
        ctl->abort = 0;
        ctl->loaded_b = -1;
        ctl->loaded_h = -1;
        tc::fence_barrier_init();
    }
    if (warp == 0) {
        tc::tmem_alloc(&ctl->tbase, TM_COLS);
        tc::tmem_relinquish();
    }
    tc::fence_proxy_async_smem();
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tbase = ctl->tbase;
    volatile int* abort = &ctl->abort;
    const uint32_t stage_tx = (uint32_t)C * 128u * (1u + (uint32_t)(R + 63) / 64u);  // xhat + bhat rows of one chunk

    if (warp == WARP_TMA) {
        // ====================================================================== TMA producer
        // The whole warp runs the loop: lane 0 arms the barriers, and the copies of a span or slot
        // are dealt out across the lanes (one copy issue costs a thread ~100 cycles).  Wait results
        // are made warp-uniform so that all lanes leave together.
        uint32_t na0 = 0, na1 = 0;  // forward-sweep uses of the two span buffers
        uint32_t slots = 0;         // per slot j: bit j = parity of its next release, bit 8 + j = release pending
        Par pr;
        bool ok = true;
        const int nbx = 1 + (R + 63) / 64;  // copies per token and chunk: xhat rows, bhat column blocks
        auto wait_all = [&](uint64_t* bar, uint32_t parity) {
            ok = __all_sync(0xffffffffu, ok && tc::mbar_wait(bar, parity, abort));
        };
        for (int it = it0; it < it1 && ok; ++it) {
            const Item I = decode_item(A, it);
            if (it > it0) wait_all(&ctl->itemdone, pr.next(B_ITEMDONE));
            if (!ok) break;
            // the item's da: 64 tokens x 4 heads per existing chunk (or this head alone, by plain
            // loads before the arrival that publishes it)
            if (!da_by_tma(P)) {
                float* ida = reinterpret_cast<float*>(sm + OFF_IDA);
                for (int i = lane; i < 2 * FL; i += 32) {
                    const int ch = i / FL, t = i % FL;
                    if (RAG ? t < (ch ? I.T[1] : I.T[0]) : I.exists[ch])  // (no read past the row's end)
                        ida[(ch * FL + t) * 4 + (I.hd & 3)] =
                            A.da[((int64_t)I.bb * P.s + (2 * I.k + ch) * FL + t) * P.heads + I.hd];
                }
                __syncwarp();
            }
            if (lane == 0) {
                uint32_t bytes = 0;
                for (int ch = 0; ch < 2; ++ch) bytes += (I.exists[ch] && da_by_tma(P)) ? 1024u : 0u;
                tc::mbar_arrive_expect_tx(&ctl->itemfull, bytes);
                for (int ch = 0; ch < 2; ++ch)
                    if (I.exists[ch] && da_by_tma(P))
                        tc::tma_load_2d(sm + OFF_IDA + ch * 1024, &tmd, I.hd & ~3, I.bb * P.s + (2 * I.k + ch) * FL,
                                        &ctl->itemfull);
            }
            // forward sweep: spans 0 .. nsp-2 alternate between the two span buffers (the last
            // one in buffer 1, so that buffer 0 frees up first for the reverse sweep)
            const int nA = (I.T[0] + SPAN - 1) / SPAN - 1;
            for (int k = 0; k < nA && ok; ++k) {
                const int b = ((nA - 1 - k) & 1) ^ 1;
                if ((b ? na1 : na0) >= 1) wait_all(&ctl->aempty[b], ((b ? na1 : na0) - 1) & 1);
                if (!ok) break;
                if (lane == 0) {
                    uint32_t by = 0;
                    for (int ch = 0; ch < 2; ++ch) by += I.exists[ch] ? SPAN * stage_tx : 0u;
                    tc::mbar_arrive_expect_tx(&ctl->afull[b], by);
                }
                __syncwarp();
                unsigned char* xb = sm + (b ? OFF_PA : OFF_SX);
                unsigned char* bt = sm + (b ? OFF_G : OFF_SB);
                for (int i = lane; i < SPAN * 2 * nbx; i += 32) {
                    const int jj = i / (2 * nbx), ch = (i / nbx) & 1, kind = i % nbx;
                    if (!I.exists[ch]) continue;
                    const int row = I.bb * P.s + (2 * I.k + ch) * FL + k * SPAN + jj;
                    if (kind == 0)
                        tc::tma_load_4d(xb + jj * 4096 + ch * 3072, &tmx, 0, I.hh, 0, row, &ctl->afull[b]);
                    else
                        tc::tma_load_4d(bt + jj * 4096 + (kind - 1) * 2048 + ch * 1024, &tmb, 64 * (kind - 1), I.hd, 0,
                                        row, &ctl->afull[b]);
                }
                if (b) ++na1; else ++na0;
            }
            // the reverse sweep's first span goes into buffer 0 once the forward sweep is done with it
            if (ok && na0 >= 1) wait_all(&ctl->aempty[0], (na0 - 1) & 1);
            if (ok) {
                // Span slots refill one by one: the reverse sweep reads slot j for the last time in
                // the d_xhat / d_bhat product of token s0 + j, so the high slots of the next span
                // load while the current span still runs on the low ones.
                const int nsp = (I.T[0] + SPAN - 1) / SPAN;
                const int ncp = nbx + (P.rw ? 1 : 0);  // copies per token and chunk
                for (int sg = nsp - 1; sg >= 0 && ok; --sg) {
                    const int s0 = sg * SPAN, len = min(SPAN, I.T[0] - s0);
                    auto slot_wait = [&](int jj) {
                        if ((slots >> (8 + jj)) & 1u) {
                            wait_all(&ctl->slotfree[jj], (slots >> jj) & 1u);
                            slots ^= (1u << jj) | (1u << (8 + jj));
                        }
                    };
                    slot_wait(len - 1);
                    // the previous span's copies must have landed before the barrier is re-armed
                    if (pr.once(U_SPAN)) wait_all(&ctl->spanfull, pr.next(B_SPAN));
                    if (!ok) break;
                    if (lane == 0) {
                        // the anchor state this span starts from, into L2 ahead of the span set-up
                        if (sg > 0)
                            tc::prefetch_l2(B.anchors + ((int64_t)blockIdx.x * NANCHOR + (sg - 1)) * 128 * 128,
                                            128u * 128u * 4u);
                        else
                            for (int ch = 0; ch < 2; ++ch)
                                if (I.exists[ch])
                                    tc::prefetch_l2(A.Hc + off_carry(P, I.bb, I.hh, 2 * I.k + ch),
                                                    (uint32_t)(P.p * P.r) * 4u);
                        uint32_t by = 0;
                        for (int ch = 0; ch < 2; ++ch)
                            if (I.exists[ch]) by += (uint32_t)len * (stage_tx + 4u * P.rw);
                        tc::mbar_arrive_expect_tx(&ctl->spanfull, by);
                    }
                    __syncwarp();
                    for (int jj = len - 1; jj >= 0 && ok; --jj) {
                        slot_wait(jj);
                        if (!ok) break;
                        slots |= 1u << (8 + jj);
                        if (lane < 2 * ncp) {
                            const int ch = lane / ncp, kind = lane % ncp;
                            if (I.exists[ch]) {
                                const int row = I.bb * P.s + (2 * I.k + ch) * FL + s0 + jj;
                                if (kind == 0)
                                    tc::tma_load_4d(sm + OFF_SX + jj * 4096 + ch * 3072, &tmx, 0, I.hh, 0, row,
                                                    &ctl->spanfull);
                                else if (kind < nbx)
                                    tc::tma_load_4d(sm + OFF_SB + jj * 4096 + (kind - 1) * 2048 + ch * 1024, &tmb, 64 * (kind - 1),
                                                    I.hd, 0, row, &ctl->spanfull);
                                else
                                    tc::tma_load_3d(sm + OFF_ROT + jj * 1024 + ch * 512, &tmr, 0, I.hd, row,
                                                    &ctl->spanfull);
                            }
                        }
                    }
                }
            }
        }
        if (!ok && lane == 0) fail(ctl, A.err, 21);
    } else if (warp == WARP_MMA) {
        // ====================================================================== MMA issuer
        if (lane == 0) {
            const uint32_t idW = tc::idesc_bf16(128, 128, 1, 1);
            const uint32_t idPre = tc::idesc_bf16(128, 128, 1, 1);
            const uint32_t idDC = tc::idesc_bf16(128, 128, 0, 0);
            const uint32_t idDX = tc::idesc_bf16(128, 16, 0, 0);
            const uint32_t idDB = tc::idesc_bf16(128, 16, 1, 0);
            const uint32_t s_g = tc::smem_u32(sm + OFF_G), s_ds = tc::smem_u32(sm + OFF_DS);
            const uint32_t s_m1t = tc::smem_u32(sm + OFF_M1T);
            const uint32_t idM1 = tc::idesc_bf16(128, 128, 0, 1);
            const uint32_t s_sx = tc::smem_u32(sm + OFF_SX), s_sb = tc::smem_u32(sm + OFF_SB);
            const uint32_t s_pa = tc::smem_u32(sm + OFF_PA);
            Par pr;
            uint32_t na0 = 0, na1 = 0, nw = 0;
            bool ok = true;
            // d_xhat / d_bhat MMAs: A = g tile (K-major rows (ch,p) / MN-major columns r), B = one
            // token's bhat / xhat tile [16 rows (8 ch + c)][128] K-major.
            auto issue_dx = [&](uint32_t sxb, uint32_t sbb) -> bool {
                if (!tc::mbar_wait(&ctl->gfull, pr.next(B_G), abort)) return false;
                if (pr.once(U_DX) && !tc::mbar_wait(&ctl->dxfree, pr.next(B_DX), abort)) return false;
                tc::tc_fence_after();
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    const uint32_t koff = (ks >> 2) * 16384u + 32u * (ks & 3);
                    const uint32_t boff = (ks >> 2) * 2048u + 32u * (ks & 3);
                    tc::mma_bf16(tbase + TM_DX, tc::sdesc_sw128(s_g + koff, 16, 1024), tc::sdesc_sw128(sbb + boff, 16, 1024),
                                 idDX, ks > 0);
                    tc::mma_bf16(tbase + TM_DB, tc::sdesc_sw128(s_g + ks * 2048u, 16384, 1024),
                                 tc::sdesc_sw128(sxb + boff, 16, 1024), idDB, ks > 0);
                }
                tc::mma_commit(&ctl->dxfull);
                tc::mma_commit(&ctl->gfree);
                return true;
            };
            auto issue_prefix = [&](int o) -> bool {
                if (!tc::mbar_wait(&ctl->pafull, pr.next(B_PA), abort)) return false;
                if (pr.once(U_PRE) && !tc::mbar_wait(&ctl->pfree, pr.next(B_P), abort)) return false;
                tc::tc_fence_after();
                // one K = 16 step per span token j <= o: A = L[t,j]-scaled xhat rows (block-diagonal
                // over the two chunks), B = the token's bhat rows
                for (int j = 0; j <= o; ++j)
                    tc::mma_bf16(tbase + TM_P, tc::sdesc_sw128(s_pa + j * 4096u, 2048, 1024),
                                 tc::sdesc_sw128(s_sb + j * 4096u, 2048, 1024), idPre, j > 0);
                tc::mma_commit(&ctl->pfull);
                tc::mma_commit(&ctl->pafree);
                return true;
            };
            auto issue_dc = [&]() -> bool {
                if (!tc::mbar_wait(&ctl->cfull, pr.next(B_C), abort)) return false;
                if (pr.once(U_DC) && !tc::mbar_wait(&ctl->dcfree, pr.next(B_DC), abort)) return false;
                tc::tc_fence_after();
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    const uint32_t koff = (ks >> 2) * 16384u + 32u * (ks & 3);
                    tc::mma_bf16_ta(tbase + TM_DC, tbase + TM_CA + 8u * ks, tc::sdesc_sw128(s_ds + koff, 16, 1024), idDC,
                                    ks > 0);
                }
                tc::mma_bf16_ta(tbase + TM_DC, tbase + TM_ONE, tc::sdesc_sw128(s_m1t, 2048, 1024), idM1, 1u);
                tc::mma_commit(&ctl->dcfull);
                tc::mma_commit(&ctl->cfree);
                return true;
            };
            for (int it = it0; it < it1 && ok; ++it) {
                const Item I = decode_item(A, it);
                // forward sweep: per span, sum_j L[end, j] W_j as one K = 8 x 16 product
                const int nA = (I.T[0] + SPAN - 1) / SPAN - 1;
                for (int k = 0; k < nA && ok; ++k) {
                    const int b = ((nA - 1 - k) & 1) ^ 1;
                    if (!(ok = tc::mbar_wait(&ctl->ascaled[b], (b ? na1 : na0) & 1, abort))) break;
                    const uint32_t wb = nw & 1;
                    if (nw >= 2 && !(ok = tc::mbar_wait(&ctl->wfree[wb], pr.next(B_W + wb), abort))) break;
                    tc::tc_fence_after();
                    const uint32_t xs = tc::smem_u32(sm + (b ? OFF_PA : OFF_SX));
                    const uint32_t bs = tc::smem_u32(sm + (b ? OFF_G : OFF_SB));
                    for (int j = 0; j < SPAN; ++j)
                        tc::mma_bf16(tbase + (wb ? TM_DC : TM_P), tc::sdesc_sw128(xs + j * 4096u, 2048, 1024),
                                     tc::sdesc_sw128(bs + j * 4096u, 2048, 1024), idW, j > 0);
                    ++nw;
                    if (b) ++na1; else ++na0;
                    tc::mma_commit(&ctl->wfull[wb]);
                    tc::mma_commit(&ctl->aempty[b]);
                }
                if (ok) {
                    const int nsp = (I.T[0] + SPAN - 1) / SPAN;
                    for (int sg = nsp - 1; sg >= 0 && ok; --sg) {
                        const int len = min(SPAN, I.T[0] - sg * SPAN);
                        // pipelined order, matching the compute warps' signals
                        for (int u = len + 1; u >= 0 && ok; --u) {
                            if (u <= len - 1) {
                                ok = issue_dx(s_sx + u * 4096u, s_sb + u * 4096u);
                                tc::mma_commit(&ctl->slotfree[u]);
                            }
                            if (ok && u - 1 >= 0 && u - 1 <= len - 1) ok = issue_dc();
                            if (ok && u - 2 >= 0) ok = issue_prefix(u - 2);
                        }
                    }
                }
            }
            if (!ok) fail(ctl, A.err, 22);
            tc::mma_commit(&ctl->fin);
            int never = 0;  // in-flight MMAs must finish before the TMEM is released
            tc::mbar_wait(&ctl->fin, 0, &never, 1u << 20);
        }
    } else {
        // ====================================================================== compute warps
        const int half = warp >> 2;
        const int m = ((warp & 3) << 5) + lane;  // TMEM lane = row (chunk, p); = r for d_bhat rows
        const int ch = m >> 6, pp = m & 63;
        const int ctid = tid;                    // 0..255
        int G[4];
        col_groups(LAYB, half, G);
        const uint32_t lane_addr = tbase + ((uint32_t)((warp & 3) * 32) << 16);
        float* acum = reinterpret_cast<float*>(sm + OFF_ACUM);            // [2][64] inclusive cumsum of da
        const float* ida = reinterpret_cast<const float*>(sm + OFF_IDA);  // [2][64][4]
        float* coefs = reinterpret_cast<float*>(sm + OFF_COEF);           // [8][2][128]
        float* Lt = reinterpret_cast<float*>(sm + OFF_LT);                // [2][8][8]
        float* myanchors = B.anchors + (int64_t)blockIdx.x * NANCHOR * 128 * 128;
        if (warp < 4) {  // the constant ONE operand: elements 0 and 1 of each row are 1
            uint32_t one[8] = {tc::pack_bf16x2(1.f, 1.f), 0u, 0u, 0u, 0u, 0u, 0u, 0u};
            tc::tmem_st8u(lane_addr + TM_ONE, one);
            tc::tmem_wait_st();
        }
        Par pr;
        uint32_t na0 = 0, na1 = 0, nw = 0;
        bool ok = true;
        for (int it = it0; it < it1; ++it) {
            const Item I = decode_item(A, it);
            const int Tch = ch ? I.T[1] : I.T[0];
            const int n = 2 * I.k + ch;
            const bool chunk_ok = ch ? I.exists[1] : I.exists[0];
            const bool half_ok = half ? I.exists[1] : I.exists[0];
            // this thread's output rows for token 0 of the item (null where it writes none): the
            // per-token steps only add the token stride
            uint64_t* ptab = reinterpret_cast<uint64_t*>(sm + OFF_PTR) + ctid * 3;
            ptab[0] = (half == 0 && chunk_ok && (!RAG || pp < P.prow))  // (past prow: zero padding rows)
                          ? reinterpret_cast<uint64_t>(B.dx + off_x(P, I.bb, n * FL, 0, I.hh) + pp)
                                              : 0ull;
            // (with row groups, d_bhat / d_rot / d_da of group g go to slice g of their buffers)
            ptab[1] = (m < R && half_ok)
                          ? reinterpret_cast<uint64_t>(B.db + I.grp * B.db_slice +
                                                       off_b(P, I.bb, (2 * I.k + half) * FL, 0, I.hd) + m)
                          : 0ull;
            // d_rot: the warp of rows 0-31 of a chunk writes its partial sums into d_rot, the warp
            // of rows 32-63 into drot2; a second pass adds the two afterwards
            ptab[2] = (P.rw > 0 && chunk_ok && n < I.proc)
                          ? reinterpret_cast<uint64_t>(((warp & 1) ? B.drot2 : B.drot) + I.grp * B.drot_slice +
                                                       off_rot(P, I.bb, n * FL, I.hd))
                          : 0ull;
            // this warp's d_da partials for its chunk (the four warps of a chunk are summed in a
            // fixed order at the end of the item, so that d_da does not depend on timing)
            float* ddap = reinterpret_cast<float*>(sm + OFF_DDA) + ch * 64 * 4 + ((warp & 1) + 2 * half);
            ok &= tc::mbar_wait(&ctl->itemfull, pr.next(B_ITEM), abort);
            // ---- item set-up: cumulative da of both chunks; D + D^T and d_m1 when (b,h) changes
            if (warp < 2) {
                const int c2 = warp;
                float* const idw = reinterpret_cast<float*>(sm + OFF_IDA);
                const float v0 = ida[(c2 * 64 + 2 * lane) * 4 + (I.hd & 3)];
                const float v1 = ida[(c2 * 64 + 2 * lane + 1) * 4 + (I.hd & 3)];
                // this head's da into slot 0 of each token's 4-head group, so that the token steps
                // read it without the head index (each lane rewrites only its own two tokens)
                idw[(c2 * 64 + 2 * lane) * 4] = v0;
                idw[(c2 * 64 + 2 * lane + 1) * 4] = v1;
                float s = v0 + v1;
#pragma unroll
                for (int off = 1; off < 32; off <<= 1) {
                    const float o2 = __shfl_up_sync(0xffffffffu, s, off);
                    if (lane >= off) s += o2;
                }
                acum[c2 * 64 + 2 * lane + 1] = s;
                acum[c2 * 64 + 2 * lane] = s - v1;
            }
            if (ctl->loaded_b != I.bb || ctl->loaded_h != I.hd) {
                const float* D = B.dm2 + ((int64_t)I.bb * P.heads + I.hd) * R * R;
                unsigned char* ds = sm + OFF_DS;
                for (int i = ctid; i < 128 * 128 / 2; i += NCW * 32) {
                    const int r2 = i >> 6, r1 = (i & 63) * 2;
                    float a0 = 0.f, a1 = 0.f;
                    if (r2 < R && r1 < R) {
                        a0 = D[(int64_t)r1 * R + r2] + D[(int64_t)r2 * R + r1];
                        a1 = D[(int64_t)(r1 + 1) * R + r2] + D[(int64_t)r2 * R + r1 + 1];
                    }
                    *reinterpret_cast<uint32_t*>(ds + tc::sw128_offset(128, r2, r1)) = tc::pack_bf16x2(a0, a1);
                }
                // d_m1 split into bf16 hi + lo rows of the K = 16 operand (rows 2..15 zero)
                const float* dm1 = B.dm1 + ((int64_t)I.bb * P.heads + I.hd) * R;
                for (int i = ctid; i < 16 * 128 / 2; i += NCW * 32) {
                    const int k = i >> 6, nn = (i & 63) * 2;
                    float v0 = 0.f, v1 = 0.f;
                    if (k < 2) {
                        const float m0 = nn < R ? dm1[nn] : 0.f, m1v = nn + 1 < R ? dm1[nn + 1] : 0.f;
                        const float h0 = __bfloat162float(__float2bfloat16_rn(m0));
                        const float h1 = __bfloat162float(__float2bfloat16_rn(m1v));
                        v0 = k == 0 ? h0 : m0 - h0;
                        v1 = k == 0 ? h1 : m1v - h1;
                    }
                    *reinterpret_cast<uint32_t*>(sm + OFF_M1T + tc::sw128_offset(16, k, nn)) = tc::pack_bf16x2(v0, v1);
                }
                tc::fence_proxy_async_smem();
            }
            named_barrier_sync(1, NCW * 32);
            if (ctid == 0) {
                if (RAG) {
                    ctl->tvalid[0] = I.T[0];
                    ctl->tvalid[1] = I.T[1];
                }
                ctl->loaded_b = I.bb;
                ctl->loaded_h = I.hd;
                for (int c2 = 0; c2 < 2; ++c2)
                    ctl->dda_row[c2] = B.dda + I.grp * B.dda_slice + off_da(P, I.bb, (2 * I.k + c2) * FL, I.hd);
            }
            const float* ac = acum + ch * 64;
            auto e_of = [&](int t) -> float { return __expf(ida[(ch * 64 + t) * 4]); };

            {
                // ================================ phase A: forward sweep, anchors
                {
                    float S[4][16];
                    if (Tch > 0) {
                        const float* src = A.Hc + off_carry(P, I.bb, I.hh, n) + (int64_t)pp * R;
#pragma unroll
                        for (int g = 0; g < 4; ++g)
#pragma unroll
                            for (int e = 0; e < 16; e += 4) {
                                const int col = 16 * G[g] + e;
                                const float4 v = col < R ? *reinterpret_cast<const float4*>(src + col)
                                                         : make_float4(0.f, 0.f, 0.f, 0.f);
                                S[g][e] = v.x; S[g][e + 1] = v.y; S[g][e + 2] = v.z; S[g][e + 3] = v.w;
                            }
                    } else {
#pragma unroll
                        for (int g = 0; g < 4; ++g)
#pragma unroll
                            for (int e = 0; e < 16; ++e) S[g][e] = 0.f;
                    }
                    // per span k: S <- D_k S + sum_j L[end, j] W_j over the span's live tokens; the
                    // tensor core forms the sum from xhat rows scaled in place by L = exp(a_end - a_j);
                    // the state after the span is anchor k
                    const int nA = (I.T[0] + SPAN - 1) / SPAN - 1;
                    // scale span k's xhat rows in place and hand them to the tensor core
                    auto scale_span = [&](int k) {
                        const int b = ((nA - 1 - k) & 1) ^ 1;
                        ok &= tc::mbar_wait(&ctl->afull[b], (b ? na1 : na0) & 1, abort);
                        unsigned char* xb = sm + (b ? OFF_PA : OFF_SX);
                        // units of 8 bf16: (token j, chunk c2, channel slot c of 4 or 8, column group jc)
                        for (int i = ctid; i < (SPAN * 16) << CS; i += NCW * 32) {
                            const int jc = i & 7, c = (i >> 3) & ((1 << CS) - 1), c2 = (i >> (3 + CS)) & 1,
                                      j = i >> (4 + CS);
                            if (c >= C) continue;
                            const int Tc = c2 ? I.T[1] : I.T[0];
                            const int t = k * SPAN + j, tend = min(k * SPAN + SPAN - 1, Tc - 1);
                            const float L = t < Tc ? __expf(acum[c2 * 64 + tend] - acum[c2 * 64 + t]) : 0.f;
                            uint4* px = reinterpret_cast<uint4*>(xb + j * 4096 + tc::sw128_chunk(16, c2, 8 * c2 + c, jc));
                            const uint4 v = *px;
                            *px = scale_bf16x8(v, L);
                        }
                        tc::fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) {
                            tc::mbar_arrive(&ctl->ascaled[b]);
                            tc::mbar_arrive(&ctl->aempty[b]);
                        }
                        if (b) ++na1; else ++na0;
                    };
                    // the next span is scaled before this span's anchor goes out, so that the
                    // anchor stores drain while the tensor core works on the next span
                    if (nA > 0) scale_span(0);
                    for (int k = 0; k < nA; ++k) {
                        const uint32_t wb = nw & 1;
                        ok &= tc::mbar_wait(&ctl->wfull[wb], pr.next(B_W + wb), abort);
                        tc::tc_fence_after();
                        const int tend = min(k * SPAN + SPAN - 1, Tch - 1);
                        const float Dk = k * SPAN < Tch ? __expf(ac[tend] - (k > 0 ? ac[k * SPAN - 1] : 0.f)) : 1.f;
#pragma unroll
                        for (int pass = 0; pass < 2; ++pass) {
                            float W[2][16];
                            tc::tmem_ld16(lane_addr + (wb ? TM_DC : TM_P) + 16 * G[2 * pass], W[0]);
                            tc::tmem_ld16(lane_addr + (wb ? TM_DC : TM_P) + 16 * G[2 * pass + 1], W[1]);
                            tc::tmem_wait_ld();
#pragma unroll
                            for (int g = 0; g < 2; ++g)
#pragma unroll
                                for (int e = 0; e < 16; e += 2)
                                    ffma2(S[2 * pass + g][e], S[2 * pass + g][e + 1], Dk, Dk, S[2 * pass + g][e],
                                          S[2 * pass + g][e + 1], W[g][e], W[g][e + 1]);
                        }
                        tc::tc_fence_before();
                        __syncwarp();
                        if (lane == 0) tc::mbar_arrive(&ctl->wfree[wb]);
                        ++nw;
                        if (k + 1 < nA) scale_span(k + 1);
                        float* dst = myanchors + (int64_t)k * 128 * 128;
#pragma unroll
                        for (int g = 0; g < 4; ++g)
#pragma unroll
                            for (int e = 0; e < 16; e += 4)
                                *reinterpret_cast<float4*>(dst + anchor_off(m, 16 * G[g] + e)) =
                                    make_float4(S[g][e], S[g][e + 1], S[g][e + 2], S[g][e + 3]);
                    }
                }
                // ================================ phase B: spans in reverse, software-pipelined
                float gr[4][16];
#pragma unroll
                for (int g = 0; g < 4; ++g)
#pragma unroll
                    for (int e = 0; e < 16; ++e) gr[g][e] = 0.f;
                float e_next = 0.f;  // e_{t+1}
                const int nsp = (I.T[0] + SPAN - 1) / SPAN;
                for (int sg = nsp - 1; sg >= 0; --sg) {
                    const int s0 = sg * SPAN, len = min(SPAN, I.T[0] - s0);
                    ok &= tc::mbar_wait(&ctl->spanfull, pr.next(B_SPAN), abort);
                    // anchor of the span -> TMEM (this thread's row and columns)
#pragma unroll
                    for (int g = 0; g < 4; ++g) {
                        float av[16];
                        const int col0 = 16 * G[g];
                        const float* carry = A.Hc + off_carry(P, I.bb, I.hh, n) + (int64_t)pp * R;
                        const float* anc = myanchors + (int64_t)(sg - 1) * 128 * 128;
                        const bool have = sg == 0 ? (Tch > 0 && col0 < R) : true;
#pragma unroll
                        for (int e = 0; e < 16; e += 4) {
                            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
                            if (have)
                                v = *reinterpret_cast<const float4*>(sg == 0 ? carry + col0 + e
                                                                           : anc + anchor_off(m, col0 + e));
                            av[e] = v.x; av[e + 1] = v.y; av[e + 2] = v.z; av[e + 3] = v.w;
                        }
                        tc::tmem_st16(lane_addr + TM_AN + col0, av);
                    }
                    tc::tmem_wait_st();
                    // decay matrix L[t, j] of the span, and cos / sin of its angles
                    if (ctid < 128) {
                        const int c2 = ctid >> 6, o = (ctid >> 3) & 7, jj = ctid & 7;
                        const float* ac2 = acum + c2 * 64;
                        Lt[ctid] = (o < len && jj <= o) ? __expf(ac2[s0 + o] - ac2[s0 + jj]) : 0.f;
                    }
                    if (ROTK == ROT_PAIRWISE || ROTK == ROT_HALF) {
                        for (int i = ctid; i < len * 2 * 64; i += NCW * 32) {
                            const int o = i >> 7, c2 = (i >> 6) & 1, a = i & 63;
                            float sv = 0.f, cv = 1.f;
                            if (a < P.na)
                                sincosf(reinterpret_cast<const float*>(sm + OFF_ROT + o * 1024 + c2 * 512)[a], &sv, &cv);
                            coefs[(o * 2 + c2) * 128 + a] = cv;
                            coefs[(o * 2 + c2) * 128 + 64 + a] = sv;
                        }
                    }
                    tc::fence_proxy_async_smem();
                    named_barrier_sync(1, NCW * 32);
                    // every thread has read its part of the span's anchor, which nothing reads again
                    // before the next item rewrites it: its 512 lines leave L2 without a write-back
                    if (sg > 0) {
                        const float* used = myanchors + ((int64_t)(sg - 1) * 128 * 128 + ctid * 64);
                        tc::discard_l2_line(used);
                        tc::discard_l2_line(used + 32);
                    }
                    const float a_anchor = s0 > 0 ? ac[s0 - 1] : 0.f;

                    // ---- prefix A tiles for token t: PA_j = L[t, s0+j] xhat_j for j <= t - s0, in the
                    // layout of the staged xhat tiles (rows 8 ch + c in column block ch); only those
                    // rows are written, the rest of the region stays zero
                    auto build_pa = [&](int t) {
                        const int o = t - s0;
                        if (pr.once(U_PA)) ok &= tc::mbar_wait(&ctl->pafree, pr.next(B_PA), abort);
                        // this thread's unit of a token row -- (chunk c2, channel slot c, 16-byte column
                        // block jc) -- is the same in every row it handles: the stride is whole rows
                        constexpr int UPR = 16 << CS;  // units per token row
                        const int u = ctid & (UPR - 1);
                        const int jc = u & 7, c = (u >> 3) & ((1 << CS) - 1), c2 = u >> (3 + CS);
                        if (c < C) {
                            const uint32_t base = tc::sw128_chunk(16, c2, 8 * c2 + c, jc);
                            const bool ex = c2 ? I.exists[1] : I.exists[0];
                            for (int j = ctid / UPR; j <= o; j += (NCW * 32) / UPR) {
                                const uint32_t off = j * 4096u + base;
                                uint4 w = make_uint4(0, 0, 0, 0);
                                if (ex) {
                                    const float L = Lt[(c2 * 8 + o) * 8 + j];
                                    const uint4 v = *reinterpret_cast<const uint4*>(sm + OFF_SX + off);
                                    w = scale_bf16x8(v, L);
                                }
                                *reinterpret_cast<uint4*>(sm + OFF_PA + off) = w;
                            }
                        }
                        tc::fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) tc::mbar_arrive(&ctl->pafull);
                    };
                    // ---- h_t from the prefix states and the anchor; d_da_{t+1}; c_t -> c tile
                    auto step_h = [&](int t) {
                        const int o = t - s0;
                        ok &= tc::mbar_wait(&ctl->pfull, pr.next(B_P), abort);
                        if (pr.once(U_C)) ok &= tc::mbar_wait(&ctl->cfree, pr.next(B_C), abort);  // CA reusable
                        tc::tc_fence_after();
                        const float dsig = __expf(ac[t] - a_anchor);
                        const bool live = t < Tch;
                        const float* cf = coefs + (o * 2 + ch) * 128;
                        const float* qt = reinterpret_cast<const float*>(sm + OFF_ROT + o * 1024 + ch * 512);
                        float dotv[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                        for (int pass = 0; pass < 2; ++pass) {
                            const int sa = slot_a<LAYB>(pass), sb = slot_b<LAYB>(pass);
                            float ha[16], hb[16], aa[16], ab[16];
                            tc::tmem_ld16(lane_addr + TM_P + 16 * G[sa], ha);
                            tc::tmem_ld16(lane_addr + TM_P + 16 * G[sb], hb);
                            tc::tmem_ld16(lane_addr + TM_AN + 16 * G[sa], aa);
                            tc::tmem_ld16(lane_addr + TM_AN + 16 * G[sb], ab);
                            tc::tmem_wait_ld();
#pragma unroll
                            for (int e = 0; e < 16; e += 2) {
                                ffma2(ha[e], ha[e + 1], dsig, dsig, aa[e], aa[e + 1], ha[e], ha[e + 1]);
                                ffma2(hb[e], hb[e + 1], dsig, dsig, ab[e], ab[e + 1], hb[e], hb[e + 1]);
                                ffma2(dotv[0], dotv[1], gr[sa][e], gr[sa][e + 1], ha[e], ha[e + 1], dotv[0], dotv[1]);
                                ffma2(dotv[2], dotv[3], gr[sb][e], gr[sb][e + 1], hb[e], hb[e + 1], dotv[2], dotv[3]);
                            }
                            rot_pass<ROTK, LAYB, false>(P, pass, 16 * G[sa], 16 * G[sb], group_rotated<ROTK>(P, G[sa]),
                                                        group_rotated<ROTK>(P, G[sb]), ha, hb, cf, qt);
                            if (live) {  // (warp-uniform: no per-word select on the common path)
                                ca_store16(lane_addr + TM_CA + 8 * G[sa], ha, false);
                                ca_store16(lane_addr + TM_CA + 8 * G[sb], hb, false);
                            } else {
                                ca_store16(lane_addr + TM_CA + 8 * G[sa], ha, true);
                                ca_store16(lane_addr + TM_CA + 8 * G[sb], hb, true);
                            }
                        }
                        tc::tmem_wait_st();
                        tc::tc_fence_before();
                        __syncwarp();
                        if (lane == 0) {
                            tc::mbar_arrive(&ctl->pfree);
                            tc::mbar_arrive(&ctl->cfull);
                        }
                        // d_da_{t+1} = e_{t+1} <g_{t+1}, h_t>  (g holds g_{t+1} here, and e_next
                        // e_{t+1}: step_g of token t+1 ran last, in this span or the one after it)
                        const float dot = warp_sum((dotv[0] + dotv[1]) + (dotv[2] + dotv[3]));
                        if (lane == 0 && t + 1 < I.T[0]) ddap[(t + 1) * 4] = e_next * dot;
                    };
                    // ---- d_c -> d_rot, G, cotangent recurrence -> g tile
                    auto step_g = [&](int t) {
                        const int o = t - s0;
                        ok &= tc::mbar_wait(&ctl->dcfull, pr.next(B_DC), abort);
                        tc::tc_fence_after();
                        const bool live = t < Tch;
                        const float* cf = coefs + (o * 2 + ch) * 128;
                        const float* qt = reinterpret_cast<const float*>(sm + OFF_ROT + o * 1024 + ch * 512);
                        const bool rot_out = ptab[2] != 0ull;
                        // this lane's d_rot partial of each pass, stored after the g tile has been
                        // handed over (its row address is formed there too, so that it is not held
                        // in registers through the passes)
                        float drv[4] = {0.f, 0.f, 0.f, 0.f};
                        int dri[4] = {-1, -1, -1, -1};  // [pass] (complex pairs), [2 pass + slot] (quaternions)
                        if (!live) {  // past valid_len: d_c = 0, so g_t = e_{t+1} g_{t+1}
                            tc::tc_fence_before();
                            __syncwarp();
                            if (lane == 0) tc::mbar_arrive(&ctl->dcfree);
#pragma unroll
                            for (int g = 0; g < 4; ++g)
#pragma unroll
                                for (int e = 0; e < 16; e += 2)
                                    fmul2(gr[g][e], gr[g][e + 1], gr[g][e], gr[g][e + 1], e_next, e_next);
                        } else {
#pragma unroll
                        for (int pass = 0; pass < 2; ++pass) {
                            const int sa = slot_a<LAYB>(pass), sb = slot_b<LAYB>(pass);
                            const bool act_a = group_rotated<ROTK>(P, G[sa]), act_b = group_rotated<ROTK>(P, G[sb]);
                            float da_[16], db_[16];
                            tc::tmem_ld16(lane_addr + TM_DC + 16 * G[sa], da_);
                            tc::tmem_ld16(lane_addr + TM_DC + 16 * G[sb], db_);
                            tc::tmem_wait_ld();  // d_c = DC: the product already added d_m1
                            // rotation-parameter gradient of the pass, summed over the warp's 32 rows
                            // by a transpose reduction (lane L then holds value L)
                            if (ROTK == ROT_PAIRWISE) {
                                if (act_b) {  // both slots hold rotated pairs
                                    float v[16];
                                    {
                                        float cc[16];
                                        ca_load16(lane_addr + TM_CA + 8 * G[sa], cc);
#pragma unroll
                                        for (int e = 0; e < 16; e += 2) v[e / 2] = da_[e] * cc[e + 1] - da_[e + 1] * cc[e];
                                    }
                                    {
                                        float cc[16];
                                        ca_load16(lane_addr + TM_CA + 8 * G[sb], cc);
#pragma unroll
                                        for (int e = 0; e < 16; e += 2)
                                            v[8 + e / 2] = db_[e] * cc[e + 1] - db_[e + 1] * cc[e];
                                    }
                                    transpose_reduce16(v, lane);
                                    const int ang = 8 * ((lane & 8) ? G[sb] : G[sa]) + (lane & 7);
                                    if (lane < 16 && ang < P.na && rot_out) { drv[pass] = v[0]; dri[pass] = ang; }
                                } else if (act_a) {
                                    float v[8];
                                    {
                                        float cc[16];
                                        ca_load16(lane_addr + TM_CA + 8 * G[sa], cc);
#pragma unroll
                                        for (int e = 0; e < 16; e += 2) v[e / 2] = da_[e] * cc[e + 1] - da_[e + 1] * cc[e];
                                    }
                                    transpose_reduce8(v, lane);
                                    const int ang = 8 * G[sa] + (lane & 7);
                                    if (lane < 8 && ang < P.na && rot_out) { drv[pass] = v[0]; dri[pass] = ang; }
                                }
                            } else if (ROTK == ROT_HALF) {
                                if (!(LAYB && pass == 1) && act_a) {
                                    float v[16];
                                    {
                                        float cc[16];
                                        ca_load16(lane_addr + TM_CA + 8 * G[sa], cc);
#pragma unroll
                                        for (int e = 0; e < 16; e += 2)
                                            fmul2(v[e], v[e + 1], -db_[e], -db_[e + 1], cc[e], cc[e + 1]);
                                    }
                                    {
                                        float cc[16];
                                        ca_load16(lane_addr + TM_CA + 8 * G[sb], cc);
#pragma unroll
                                        for (int e = 0; e < 16; e += 2)
                                            ffma2(v[e], v[e + 1], da_[e], da_[e + 1], cc[e], cc[e + 1], v[e], v[e + 1]);
                                    }
                                    transpose_reduce16(v, lane);
                                    const int ang = 16 * G[sa] + (lane & 15);
                                    if (lane < 16 && ang < P.na && rot_out) { drv[pass] = v[0]; dri[pass] = ang; }
                                }
                            } else if (ROTK == ROT_QUAT) {
                                // sum_p d_c (x) conj(c) per 4-block; the factor (.) (x) Q / |Q|^2, linear,
                                // is applied once the two row halves' partial sums are added
#pragma unroll
                                for (int sl = 0; sl < 2; ++sl) {
                                    if (!(sl ? act_b : act_a)) continue;
                                    const int gsl = sl ? sb : sa;
                                    float v[16];
                                    {
                                        float cc[16];
                                        ca_load16(lane_addr + TM_CA + 8 * G[gsl], cc);
                                        const float(&d)[16] = sl ? db_ : da_;
#pragma unroll
                                        for (int bq = 0; bq < 4; ++bq)
                                            hamilton(d[4 * bq], d[4 * bq + 1], d[4 * bq + 2], d[4 * bq + 3], cc[4 * bq],
                                                     -cc[4 * bq + 1], -cc[4 * bq + 2], -cc[4 * bq + 3], v[4 * bq],
                                                     v[4 * bq + 1], v[4 * bq + 2], v[4 * bq + 3]);
                                    }
                                    transpose_reduce16(v, lane);
                                    // lanes 4i..4i+3 (i < 4) hold the 4 components of block i
                                    const int blk = 4 * G[gsl] + ((lane >> 2) & 3);
                                    if (lane < 16 && blk < P.J && rot_out) {
                                        drv[2 * pass + sl] = v[0];
                                        dri[2 * pass + sl] = 4 * blk + (lane & 3);
                                    }
                                }
                            }
                            // G = derot^T(d_c); g_t = G_t + e_{t+1} g_{t+1}
                            rot_pass<ROTK, LAYB, true>(P, pass, 16 * G[sa], 16 * G[sb], act_a, act_b, da_, db_, cf, qt);
#pragma unroll
                            for (int e = 0; e < 16; e += 2) {
                                ffma2(gr[sa][e], gr[sa][e + 1], e_next, e_next, gr[sa][e], gr[sa][e + 1], da_[e], da_[e + 1]);
                                ffma2(gr[sb][e], gr[sb][e + 1], e_next, e_next, gr[sb][e], gr[sb][e + 1], db_[e], db_[e + 1]);
                            }
                        }
                        tc::tc_fence_before();
                        __syncwarp();
                        if (lane == 0) tc::mbar_arrive(&ctl->dcfree);
                        }
                        e_next = e_of(t);
                        if (pr.once(U_G)) ok &= tc::mbar_wait(&ctl->gfree, pr.next(B_G), abort);
#pragma unroll
                        for (int g = 0; g < 4; ++g) write_tile16(sm + OFF_G, m, G[g], gr[g], false);
                        tc::fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) tc::mbar_arrive(&ctl->gfull);
                        if (rot_out && (!RAG || live)) {  // the row address only now, not held through the passes
                            float* const drot_t = reinterpret_cast<float*>(ptab[2]) + (int64_t)t * P.heads * P.rw;
#pragma unroll
                            for (int k = 0; k < 4; ++k)
                                if (dri[k] >= 0) drot_t[dri[k]] = drv[k];
                        }
                    };
                    // ---- d_xhat (lanes = rows) and d_bhat (lanes = r) of token t
                    auto step_out = [&](int t) {
                        ok &= tc::mbar_wait(&ctl->dxfull, pr.next(B_DX), abort);
                        tc::tc_fence_after();
                        float v[8], u[8];
                        tc::tmem_ld8(lane_addr + TM_DX + 8 * ch, v);
                        tc::tmem_ld8(lane_addr + TM_DB + 8 * half, u);
                        tc::tmem_wait_ld();
                        tc::tc_fence_before();
                        __syncwarp();
                        if (lane == 0) tc::mbar_arrive(&ctl->dxfree);
                        const int64_t hp = (int64_t)P.h * (RAG ? P.prow : P.p), hr = (int64_t)P.heads * P.r;
                        if (ptab[0] && (!RAG || t < Tch)) {
                            __nv_bfloat16* px = reinterpret_cast<__nv_bfloat16*>(ptab[0]) + (int64_t)t * C * hp;
#pragma unroll
                            for (int c = 0; c < (1 << CS); ++c)
                                if (c < C) px[c * hp] = __float2bfloat16_rn(v[c]);
                        }
                        if (ptab[1] && (!RAG || t < ctl->tvalid[half])) {
                            __nv_bfloat16* pb = reinterpret_cast<__nv_bfloat16*>(ptab[1]) + (int64_t)t * C * hr;
#pragma unroll
                            for (int c = 0; c < (1 << CS); ++c)
                                if (c < C) pb[c * hr] = __float2bfloat16_rn(u[c]);
                        }
                    };

                    // u runs two tokens ahead so that every step has one call site
                    const int thi = s0 + len - 1;
                    for (int u = thi + 2; u >= s0; --u) {
                        if (u <= thi) step_g(u);
                        if (u - 1 >= s0 && u - 1 <= thi) step_h(u - 1);
                        if (u - 2 >= s0) build_pa(u - 2);
                        if (u <= thi) step_out(u);
                    }
                }
                // ---- chunk start: d_da_0 = e_0 <g_0, h_->, e_n = e_0 g_0 (anchor 0 = the carry)
                {
                    float dot = 0.f;
#pragma unroll
                    for (int g = 0; g < 4; ++g) {
                        float an[16];
                        tc::tmem_ld16(lane_addr + TM_AN + 16 * G[g], an);
                        tc::tmem_wait_ld();
#pragma unroll
                        for (int e = 0; e < 16; ++e) dot = fmaf(gr[g][e], an[e], dot);
                    }
                    dot = warp_sum(dot);
                    if (lane == 0 && Tch > 0) ddap[0] = e_of(0) * dot;
                    if (Tch > 0) {
                        const float e0 = e_of(0);
                        float* dst = B.E + off_carry(P, I.bb, I.hh, n) + (int64_t)pp * R;
#pragma unroll
                        for (int g = 0; g < 4; ++g)
#pragma unroll
                            for (int e = 0; e < 16; e += 4) {
                                const int col = 16 * G[g] + e;
                                if (col < R)
                                    *reinterpret_cast<float4*>(dst + col) = make_float4(
                                        e0 * gr[g][e], e0 * gr[g][e + 1], e0 * gr[g][e + 2], e0 * gr[g][e + 3]);
                            }
                    }
                }
            }
            // ---- d_da of the item's valid tokens: the four warps' partials of each chunk, in order
            named_barrier_sync(2, NCW * 32);
            if (ctid < 128) {
                const int c2 = ctid >> 6, t = ctid & 63, n2 = 2 * I.k + c2;
                const int T2 = c2 ? I.T[1] : I.T[0];
                if (t < T2 && n2 < I.proc) {
                    const float* pq = reinterpret_cast<const float*>(sm + OFF_DDA) + (c2 * 64 + t) * 4;
                    ctl->dda_row[c2][(int64_t)t * P.heads] = ((pq[0] + pq[1]) + pq[2]) + pq[3];
                }
            }
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&ctl->itemdone);
        }
        if (!ok) fail(ctl, A.err, 23);
    }
    // ---- teardown
    tc::tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc::tc_fence_after();
        tc::tmem_dealloc(tbase, TM_COLS);
    }
}

// the general-shape kernel (RAG: partial last chunks, fewer than 64 rows), compiled in fast_bwd_rag.cu
using BwdKernel = decltype(&tc_bwd_kernel<ROT_NONE, 0, 2, false>);
BwdKernel ragged_bwd_kernel(int rot, int layoutB, bool c8);

}  // namespace fastbwd
