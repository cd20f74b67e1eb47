// fast_bwd.cu -- tcgen05 / TMA recompute backward of the state-moments operator (bf16 operands,
// p = 64, r in {64, 128}, C <= 4).
//
// Work item = a pair of 64-token chunks of one (batch row, head); the two chunks share the 128
// TMEM lanes (row m = (chunk, p)) as in the forward.  Two modes:
//
// LOCAL  -- the chunk's own backward with zero incoming carry cotangent ("backward.rs", module
//   header "Gradient math", with the d_h+ term split off):
//   phase A  forward sweep h = e^{da} h + W from the chunk carry (W by one block-diagonal MMA per
//            token); the state after every 8th token is kept as an fp32 anchor in this CTA's
//            workspace slot (7 anchors; the chunk carry is anchor 0).
//   phase B  8-token spans in reverse.  For token t of a span starting at s0 the state is
//            rebuilt exactly as  h_t = (prod_{s0<=i<=t} e_i) A + sum_{s0<=j<=t} L[t,j] W_j : one
//            prefix MMA whose A rows are xhat rows scaled by L[t,j] = exp(a_t - a_j) (two tokens
//            per K=16 step), plus the anchor term read from TMEM.  Then c = derot(h) (bf16 tile),
//            d_c = c (D + D^T) + d_m1 on tcgen05 (K = r), d_rot from (c, d_c) by warp transpose
//            reductions over p, G = derot^T(d_c), the cotangent recurrence g_t = G_t + e_{t+1}
//            g_{t+1} in registers, d_da_{t+1} = e_{t+1} <g_{t+1}, h_t>, and d_xhat = g bhat^T,
//            d_bhat = g^T xhat as N = 16 MMAs.  After the chunk: e_n = e_0 g_0.
// CORR   -- adds the carry cotangent dH = dH(n+1) of every chunk but the last processed one:
//   d_xhat_jc += sc_j dH bhat_jc, d_bhat_jc += sc_j dH^T xhat_jc (the same N = 16 MMAs with the
//   constant bf16 dH tile), d_da_s += D_n <dH, h_-> + sum_{j<s} sc_j <dH, W_j>, sc_j = e^{a_last-a_j}.
//
// Warp roles: 0-7 compute (two threads per row, 64 columns each), 8 TMA, 9 MMA.  Every wait is
// bounded; a timeout sets the workspace error word and the CTA winds down.
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
constexpr int NS = 4;          // forward-sweep / correction staging ring (in the prefix tiles' space)
constexpr int SPAN = 8;        // tokens per anchor span
constexpr int NANCHOR = 7;     // anchors per 64-token chunk kept in the workspace (anchor 0 = carry)

// shared memory map (bytes from a 1024-aligned base)
constexpr uint32_t OFF_C = 0;                    // c tile     [128 rows (ch,p)][128 r] bf16, 32 KB
constexpr uint32_t OFF_G = 32768;                // g tile     (same layout)
constexpr uint32_t OFF_DS = 65536;               // D + D^T    [128 r2][128 r1] bf16
constexpr uint32_t OFF_SX = 98304;               // span xhat tiles, 8 x [16 rows (8ch+c)][128 (ch,p)]
constexpr uint32_t OFF_SB = 131072;              // span bhat tiles, 8 x [16 rows (8ch+c)][128 r]
constexpr uint32_t OFF_PB = 163840;              // prefix B   [64 rows (8jj+4ch+c)][128 r]
constexpr uint32_t OFF_PA = 180224;              // prefix A   [64 rows][128 (ch,p)]
constexpr uint32_t OFF_RING = OFF_PB;            // ring stage s: X at +8 KB s, B at +8 KB s + 4 KB
constexpr uint32_t OFF_ROT = 196608;             // span rotation rows, 8 tokens x 2 chunks x 512 B
constexpr uint32_t OFF_IDA = 204800;             // item da: 2 chunks x 64 tokens x 4 heads fp32
constexpr uint32_t OFF_ACUM = 206848;            // cumulative da, 2 chunks x 64 fp32
constexpr uint32_t OFF_COEF = 207360;            // 2 bufs x 2 chunks x 256 fp32 (cos | sin)
constexpr uint32_t OFF_M1 = 211456;              // d_m1 [128] fp32
constexpr uint32_t OFF_RED = 211968;             // 2 bufs x 2 chunks x 128 fp32 d_rot partials
constexpr uint32_t OFF_RDA = 214016;             // 2 bufs x 2 chunks fp32 d_da partials (+ pad)
constexpr uint32_t OFF_OM = 214144;              // correction: 2 chunks x 64 fp32 omega_j
constexpr uint32_t OFF_BASE = 214656;            // correction: 2 chunks fp32 base terms (+ pad)
constexpr uint32_t OFF_CTL = 214784;
constexpr uint32_t SMEM_BYTES = OFF_CTL + 512 + 1024;
static_assert(OFF_SX % 1024 == 0 && OFF_SB % 1024 == 0 && OFF_PB % 1024 == 0 && OFF_PA % 1024 == 0, "tiles");
static_assert(OFF_ROT % 128 == 0 && OFF_IDA % 128 == 0 && OFF_CTL % 8 == 0, "tensor-copy slots");
static_assert(SMEM_BYTES <= 232448, "shared memory");

struct Ctl {
    uint64_t itemfull, itemdone;
    uint64_t full[NS], empty[NS];
    uint64_t wfull[2], wfree[2];
    uint64_t spanfull, spanfree, pbready;
    uint64_t pafull, pafree, pfull, pfree;
    uint64_t cfull, cfree, dcfull, dcfree;
    uint64_t gfull, gfree, dxfull, dxfree;
    uint64_t fin;
    uint32_t tbase;
    int abort;
    int loaded_b, loaded_h;
};
static_assert(sizeof(Ctl) <= 512, "control block");

// tensor memory columns
constexpr uint32_t TM_P = 0, TM_DC = 128, TM_AN = 256, TM_DX = 384, TM_DB = 400, TM_COLS = 512;

enum { LOCAL = 0, CORR = 1 };

struct BwdArgs {
    FastArgs F;         // problem, items, Hc (carries), Dn, err
    float* E;           // [b,h,nc,p,r]: LOCAL writes e_n; CORR reads dH(n+1)
    float* anchors;     // [grid][7][128][128] fp32 anchor slots
    const float* dm2;   // [b,h,r,r]
    const float* dm1;   // [b,h,r]
    __nv_bfloat16* dx;  // d_xhat
    __nv_bfloat16* db;  // d_bhat
    float* dda;         // d_da
    float* drot;        // d_rot
};

__device__ __forceinline__ void fail(Ctl* ctl, int* err, int code) {
    ctl->abort = 1;
    atomicExch(err, code);
}

// Sum of 32 per-lane values across the warp, transposed: on return v[0] of lane L holds the sum
// over all lanes of the original v[L].
__device__ __forceinline__ void transpose_reduce32(float (&v)[32], int lane) {
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) {
        const bool upper = (lane & off) != 0;
#pragma unroll
        for (int i = 0; i < off; ++i) {
            const float send = upper ? v[i] : v[i + off];
            const float keep = upper ? v[i + off] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
        }
    }
}

__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Read this thread's 64 columns of row m of a bf16 [128 x 128] swizzled tile as floats.
__device__ __forceinline__ void read_tile_row(const unsigned char* tile, int m, const int (&G)[4],
                                              float (&v)[4][16]) {
#pragma unroll
    for (int g = 0; g < 4; ++g) {
        const uint32_t hv = G[g] >> 2, j0 = 2 * (G[g] & 3);
#pragma unroll
        for (int hj = 0; hj < 2; ++hj) {
            const uint4 w = *reinterpret_cast<const uint4*>(tile + tc::sw128_chunk(128, hv, m, j0 + hj));
            v[g][8 * hj + 0] = bf16lo(w.x); v[g][8 * hj + 1] = bf16hi(w.x);
            v[g][8 * hj + 2] = bf16lo(w.y); v[g][8 * hj + 3] = bf16hi(w.y);
            v[g][8 * hj + 4] = bf16lo(w.z); v[g][8 * hj + 5] = bf16hi(w.z);
            v[g][8 * hj + 6] = bf16lo(w.w); v[g][8 * hj + 7] = bf16hi(w.w);
        }
    }
}
__device__ __forceinline__ void write_tile_row(unsigned char* tile, int m, const int (&G)[4], const float (&v)[4][16],
                                               bool zero) {
#pragma unroll
    for (int g = 0; g < 4; ++g) {
        const uint32_t hv = G[g] >> 2, j0 = 2 * (G[g] & 3);
#pragma unroll
        for (int hj = 0; hj < 2; ++hj) {
            uint4 w = make_uint4(0, 0, 0, 0);
            if (!zero) {
                w.x = tc::pack_bf16x2(v[g][8 * hj + 0], v[g][8 * hj + 1]);
                w.y = tc::pack_bf16x2(v[g][8 * hj + 2], v[g][8 * hj + 3]);
                w.z = tc::pack_bf16x2(v[g][8 * hj + 4], v[g][8 * hj + 5]);
                w.w = tc::pack_bf16x2(v[g][8 * hj + 6], v[g][8 * hj + 7]);
            }
            *reinterpret_cast<uint4*>(tile + tc::sw128_chunk(128, hv, m, j0 + hj)) = w;
        }
    }
}
__device__ __forceinline__ void tmem_ld_row(uint32_t addr, const int (&G)[4], float (&v)[4][16]) {
#pragma unroll
    for (int g = 0; g < 4; ++g) tc::tmem_ld16(addr + 16 * G[g], v[g]);
    tc::tmem_wait_ld();
}

// Parity helpers: a barrier that completes once per use; `n` = number of completed uses waited so far.
struct Phase {
    uint32_t n = 0;
    __device__ uint32_t next() { return (n++) & 1; }
};

template <int MODE>
__global__ void __launch_bounds__(NTHR, 1)
    tc_bwd_kernel(const __grid_constant__ BwdArgs B, const __grid_constant__ CUtensorMap tmx,
                  const __grid_constant__ CUtensorMap tmb, const __grid_constant__ CUtensorMap tmr,
                  const __grid_constant__ CUtensorMap tmd) {
    extern __shared__ unsigned char smraw[];
    unsigned char* sm = (unsigned char*)(((uintptr_t)smraw + 1023) & ~(uintptr_t)1023);
    Ctl* ctl = reinterpret_cast<Ctl*>(sm + OFF_CTL);
    const FastArgs& A = B.F;
    const MMParams& P = A.P;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int R = P.r, C = P.C;
    const int it0 = item_begin(A, blockIdx.x), it1 = item_begin(A, blockIdx.x + 1);

    // ---- set-up: zero the operand tiles whose padding rows/halves must read as zero
    for (uint32_t i = tid; i < (OFF_ROT - OFF_C) / 16; i += NTHR)
        reinterpret_cast<uint4*>(sm + OFF_C)[i] = make_uint4(0, 0, 0, 0);
    for (uint32_t i = tid; i < (OFF_CTL - OFF_ROT) / 4; i += NTHR) reinterpret_cast<float*>(sm + OFF_ROT)[i] = 0.f;
    if (tid == 0) {
        tc::mbar_init(&ctl->itemfull, 1);
        tc::mbar_init(&ctl->itemdone, NCW);
        for (int s = 0; s < NS; ++s) {
            tc::mbar_init(&ctl->full[s], 1);
            tc::mbar_init(&ctl->empty[s], 1 + NCW);
        }
        for (int i = 0; i < 2; ++i) {
            tc::mbar_init(&ctl->wfull[i], 1);
            tc::mbar_init(&ctl->wfree[i], NCW);
        }
        tc::mbar_init(&ctl->spanfull, 1);
        tc::mbar_init(&ctl->spanfree, 1 + NCW);
        tc::mbar_init(&ctl->pbready, NCW);
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
    const uint32_t stage_tx = (uint32_t)C * 128u * (1u + (uint32_t)R / 64u);  // xhat + bhat rows of one chunk

    if (warp == WARP_TMA) {
        // ====================================================================== TMA producer
        if (lane == 0) {
            uint32_t q = 0;  // ring uses
            Phase ph_itemdone, ph_spanfree;
            uint32_t spans_done = 0;
            bool ok = true;
            for (int it = it0; it < it1 && ok; ++it) {
                const Item I = decode_item(A, it);
                if (it > it0) ok &= tc::mbar_wait(&ctl->itemdone, ph_itemdone.next(), abort);
                if (!ok) break;
                // the item's da: 64 tokens x 4 heads per existing chunk
                uint32_t bytes = 0;
                for (int ch = 0; ch < 2; ++ch) bytes += I.exists[ch] ? 1024u : 0u;
                tc::mbar_arrive_expect_tx(&ctl->itemfull, bytes);
                for (int ch = 0; ch < 2; ++ch)
                    if (I.exists[ch])
                        tc::tma_load_2d(sm + OFF_IDA + ch * 1024, &tmd, I.hh & ~3, I.bb * P.s + (2 * I.k + ch) * FL,
                                        &ctl->itemfull);
                // forward sweep (LOCAL) / correction tokens (CORR) through the ring
                for (int t = 0; t < I.T[0] && ok; ++t, ++q) {
                    const uint32_t s = q % NS, u = q / NS;
                    if (u >= 1) ok &= tc::mbar_wait(&ctl->empty[s], (u - 1) & 1, abort);
                    if (!ok) break;
                    uint32_t by = 0;
                    for (int ch = 0; ch < 2; ++ch) by += I.exists[ch] ? stage_tx : 0u;
                    tc::mbar_arrive_expect_tx(&ctl->full[s], by);
                    unsigned char* st = sm + OFF_RING + s * 8192;
                    for (int ch = 0; ch < 2; ++ch) {
                        if (!I.exists[ch]) continue;
                        const int row = I.bb * P.s + (2 * I.k + ch) * FL + t;
                        tc::tma_load_4d(st + ch * 3072, &tmx, 0, I.hh, 0, row, &ctl->full[s]);
                        for (int a = 0; a < R / 64; ++a)
                            tc::tma_load_5d(st + 4096 + a * 2048 + ch * 1024, &tmb, 0, a, I.hh, 0, row, &ctl->full[s]);
                    }
                }
                if (MODE == LOCAL && ok) {
                    const int nsp = (I.T[0] + SPAN - 1) / SPAN;
                    for (int sg = nsp - 1; sg >= 0 && ok; --sg) {
                        if (spans_done >= 1) ok &= tc::mbar_wait(&ctl->spanfree, ph_spanfree.next(), abort);
                        if (!ok) break;
                        const int s0 = sg * SPAN, len = min(SPAN, I.T[0] - s0);
                        uint32_t by = 0;
                        for (int ch = 0; ch < 2; ++ch)
                            if (I.exists[ch]) by += (uint32_t)len * (stage_tx + 4u * P.rw);
                        tc::mbar_arrive_expect_tx(&ctl->spanfull, by);
                        for (int jj = 0; jj < len; ++jj)
                            for (int ch = 0; ch < 2; ++ch) {
                                if (!I.exists[ch]) continue;
                                const int row = I.bb * P.s + (2 * I.k + ch) * FL + s0 + jj;
                                tc::tma_load_4d(sm + OFF_SX + jj * 4096 + ch * 3072, &tmx, 0, I.hh, 0, row,
                                                &ctl->spanfull);
                                for (int a = 0; a < R / 64; ++a)
                                    tc::tma_load_5d(sm + OFF_SB + jj * 4096 + a * 2048 + ch * 1024, &tmb, 0, a, I.hh,
                                                    0, row, &ctl->spanfull);
                                if (P.rw)
                                    tc::tma_load_3d(sm + OFF_ROT + jj * 1024 + ch * 512, &tmr, 0, I.hh, row,
                                                    &ctl->spanfull);
                            }
                        ++spans_done;
                    }
                }
            }
            if (!ok) fail(ctl, A.err, 21);
        }
    } else if (warp == WARP_MMA) {
        // ====================================================================== MMA issuer
        if (lane == 0) {
            const uint32_t idW = tc::idesc_bf16(128, 128, 1, 1);
            const uint32_t idPre = tc::idesc_bf16(128, 128, 1, 1);
            const uint32_t idDC = tc::idesc_bf16(128, 128, 0, 0);
            const uint32_t idDX = tc::idesc_bf16(128, 16, 0, 0);
            const uint32_t idDB = tc::idesc_bf16(128, 16, 1, 0);
            const uint32_t s_ring = tc::smem_u32(sm + OFF_RING), s_c = tc::smem_u32(sm + OFF_C);
            const uint32_t s_g = tc::smem_u32(sm + OFF_G), s_ds = tc::smem_u32(sm + OFF_DS);
            const uint32_t s_sx = tc::smem_u32(sm + OFF_SX), s_sb = tc::smem_u32(sm + OFF_SB);
            const uint32_t s_pa = tc::smem_u32(sm + OFF_PA), s_pb = tc::smem_u32(sm + OFF_PB);
            Phase ph_full[NS], ph_wfree[2], ph_pbready, ph_pafull, ph_pfree, ph_cfull, ph_dcfree, ph_gfull, ph_dxfree;
            uint32_t q = 0, nw = 0, npre = 0, ndc = 0, ndx = 0;
            bool ok = true;
            // d_xhat / d_bhat MMAs: A = g tile (K-major rows (ch,p) / MN-major columns r), B = one
            // token's bhat / xhat tile [16 rows (8 ch + c)][128] K-major.
            auto issue_dx = [&](uint32_t sxb, uint32_t sbb, bool wait_g, bool free_g) -> bool {
                if (wait_g && !tc::mbar_wait(&ctl->gfull, ph_gfull.next(), abort)) return false;
                if (ndx >= 1 && !tc::mbar_wait(&ctl->dxfree, ph_dxfree.next(), abort)) return false;
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
                ++ndx;
                tc::mma_commit(&ctl->dxfull);
                if (free_g) tc::mma_commit(&ctl->gfree);
                return true;
            };
            for (int it = it0; it < it1 && ok; ++it) {
                const Item I = decode_item(A, it);
                for (int t = 0; t < I.T[0] && ok; ++t, ++q) {
                    const uint32_t s = q % NS;
                    const uint32_t xb = s_ring + s * 8192, bb_ = xb + 4096;
                    if (!(ok = tc::mbar_wait(&ctl->full[s], ph_full[s].next(), abort))) break;
                    if (MODE == LOCAL) {
                        const uint32_t wb = nw & 1;
                        if (nw >= 2 && !(ok = tc::mbar_wait(&ctl->wfree[wb], ph_wfree[wb].next(), abort))) break;
                        tc::tc_fence_after();
                        tc::mma_bf16(tbase + (wb ? TM_DC : TM_P), tc::sdesc_sw128(xb, 2048, 1024),
                                     tc::sdesc_sw128(bb_, 2048, 1024), idW, 0);
                        ++nw;
                        tc::mma_commit(&ctl->wfull[wb]);
                        tc::mma_commit(&ctl->empty[s]);
                    } else {
                        if (!(ok = issue_dx(xb, bb_, t == 0, t == I.T[0] - 1))) break;
                        tc::mma_commit(&ctl->empty[s]);
                    }
                }
                if (MODE == LOCAL && ok) {
                    const int nsp = (I.T[0] + SPAN - 1) / SPAN;
                    for (int sg = nsp - 1; sg >= 0 && ok; --sg) {
                        const int s0 = sg * SPAN, len = min(SPAN, I.T[0] - s0);
                        if (!(ok = tc::mbar_wait(&ctl->pbready, ph_pbready.next(), abort))) break;
                        for (int o = len - 1; o >= 0 && ok; --o) {
                            // prefix states of token s0 + o
                            if (!(ok = tc::mbar_wait(&ctl->pafull, ph_pafull.next(), abort))) break;
                            if (npre >= 1 && !(ok = tc::mbar_wait(&ctl->pfree, ph_pfree.next(), abort))) break;
                            tc::tc_fence_after();
                            const int nk = o / 2 + 1;
                            for (int kq = 0; kq < nk; ++kq)
                                tc::mma_bf16(tbase + TM_P, tc::sdesc_sw128(s_pa + kq * 2048u, 8192, 1024),
                                             tc::sdesc_sw128(s_pb + kq * 2048u, 8192, 1024), idPre, kq > 0);
                            ++npre;
                            tc::mma_commit(&ctl->pfull);
                            tc::mma_commit(&ctl->pafree);
                            // moments VJP d_c = c (D + D^T)
                            if (!(ok = tc::mbar_wait(&ctl->cfull, ph_cfull.next(), abort))) break;
                            if (ndc >= 1 && !(ok = tc::mbar_wait(&ctl->dcfree, ph_dcfree.next(), abort))) break;
                            tc::tc_fence_after();
#pragma unroll
                            for (int ks = 0; ks < 8; ++ks) {
                                const uint32_t koff = (ks >> 2) * 16384u + 32u * (ks & 3);
                                tc::mma_bf16(tbase + TM_DC, tc::sdesc_sw128(s_c + koff, 16, 1024),
                                             tc::sdesc_sw128(s_ds + koff, 16, 1024), idDC, ks > 0);
                            }
                            ++ndc;
                            tc::mma_commit(&ctl->dcfull);
                            tc::mma_commit(&ctl->cfree);
                            // d_xhat / d_bhat of the token
                            if (!(ok = issue_dx(s_sx + o * 4096u, s_sb + o * 4096u, true, true))) break;
                        }
                        if (ok) tc::mma_commit(&ctl->spanfree);
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
        col_groups(A.layoutB, half, G);
        const uint32_t lane_addr = tbase + ((uint32_t)((warp & 3) * 32) << 16);
        float* acum = reinterpret_cast<float*>(sm + OFF_ACUM);   // [2][64] inclusive cumsum of da
        const float* ida = reinterpret_cast<const float*>(sm + OFF_IDA);  // [2][64][4]
        float* m1s = reinterpret_cast<float*>(sm + OFF_M1);
        float* red = reinterpret_cast<float*>(sm + OFF_RED);     // [2 bufs][2 ch][128]
        float* rda = reinterpret_cast<float*>(sm + OFF_RDA);     // [2 bufs][2 ch]
        float* om = reinterpret_cast<float*>(sm + OFF_OM);       // [2 ch][64]
        float* base = reinterpret_cast<float*>(sm + OFF_BASE);   // [2 ch]
        float* myanchors = B.anchors + (int64_t)blockIdx.x * NANCHOR * 128 * 128;
        Phase ph_itemfull, ph_full[NS], ph_wfull[2], ph_spanfull, ph_pfull, ph_pafree, ph_cfree, ph_dcfull, ph_gfree,
            ph_dxfull;
        uint32_t q = 0, nw = 0, npa = 0, nc_ = 0, ng = 0;
        bool ok = true;
        for (int it = it0; it < it1; ++it) {
            const Item I = decode_item(A, it);
            const int Tch = I.T[ch];
            const int n = 2 * I.k + ch;
            const bool chunk_ok = I.exists[ch];
            ok &= tc::mbar_wait(&ctl->itemfull, ph_itemfull.next(), abort);
            // ---- item set-up: cumulative da of both chunks; D + D^T and d_m1 when (b,h) changes
            if (warp < 2) {
                const int c2 = warp;
                float v0 = ida[(c2 * 64 + 2 * lane) * 4 + (I.hh & 3)];
                float v1 = ida[(c2 * 64 + 2 * lane + 1) * 4 + (I.hh & 3)];
                float s = v0 + v1;
#pragma unroll
                for (int off = 1; off < 32; off <<= 1) {
                    const float o2 = __shfl_up_sync(0xffffffffu, s, off);
                    if (lane >= off) s += o2;
                }
                acum[c2 * 64 + 2 * lane + 1] = s;
                acum[c2 * 64 + 2 * lane] = s - v1;
            }
            if (MODE == LOCAL && (ctl->loaded_b != I.bb || ctl->loaded_h != I.hh)) {
                const float* D = B.dm2 + ((int64_t)I.bb * P.h + I.hh) * R * R;
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
                for (int i = ctid; i < 128; i += NCW * 32)
                    m1s[i] = i < R ? B.dm1[((int64_t)I.bb * P.h + I.hh) * R + i] : 0.f;
                tc::fence_proxy_async_smem();
            }
            named_barrier_sync(1, NCW * 32);
            if (MODE == LOCAL && ctid == 0) {
                ctl->loaded_b = I.bb;
                ctl->loaded_h = I.hh;
            }
            const float* ac = acum + ch * 64;
            auto e_of = [&](int t) -> float { return __expf(ida[(ch * 64 + t) * 4 + (I.hh & 3)]); };

            if (MODE == LOCAL) {
                // ================================ phase A: forward sweep, anchors
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
                for (int t = 0; t < I.T[0]; ++t, ++q) {
                    const uint32_t s = q % NS, wb = nw & 1;
                    ok &= tc::mbar_wait(&ctl->full[s], ph_full[s].next(), abort);
                    ok &= tc::mbar_wait(&ctl->wfull[wb], ph_wfull[wb].next(), abort);
                    tc::tc_fence_after();
                    float W[4][16];
                    tmem_ld_row(lane_addr + (wb ? TM_DC : TM_P), G, W);
                    tc::tc_fence_before();
                    __syncwarp();
                    if (lane == 0) {
                        tc::mbar_arrive(&ctl->wfree[wb]);
                        tc::mbar_arrive(&ctl->empty[s]);
                    }
                    ++nw;
                    if (t < Tch) {
                        const float et = e_of(t);
#pragma unroll
                        for (int g = 0; g < 4; ++g)
#pragma unroll
                            for (int e = 0; e < 16; ++e) S[g][e] = fmaf(et, S[g][e], W[g][e]);
                    }
                    if ((t + 1) % SPAN == 0 && t + 1 < I.T[0]) {  // anchor of the span starting at t + 1
                        float* dst = myanchors + ((int64_t)((t + 1) / SPAN - 1) * 128 + m) * 128;
#pragma unroll
                        for (int g = 0; g < 4; ++g)
#pragma unroll
                            for (int e = 0; e < 16; e += 4)
                                *reinterpret_cast<float4*>(dst + 16 * G[g] + e) =
                                    make_float4(S[g][e], S[g][e + 1], S[g][e + 2], S[g][e + 3]);
                    }
                }
                // ================================ phase B: spans in reverse
                float gr[4][16];
#pragma unroll
                for (int g = 0; g < 4; ++g)
#pragma unroll
                    for (int e = 0; e < 16; ++e) gr[g][e] = 0.f;
                float e_next = 0.f;  // e_{t+1}
                const int nsp = (I.T[0] + SPAN - 1) / SPAN;
                for (int sg = nsp - 1; sg >= 0; --sg) {
                    const int s0 = sg * SPAN, len = min(SPAN, I.T[0] - s0);
                    ok &= tc::mbar_wait(&ctl->spanfull, ph_spanfull.next(), abort);
                    // anchor of the span -> TMEM (this thread's row and columns)
                    {
                        float av[4][16];
                        const float* src = sg == 0 ? (A.Hc + off_carry(P, I.bb, I.hh, n) + (int64_t)pp * R)
                                                   : (myanchors + ((int64_t)(sg - 1) * 128 + m) * 128);
                        const bool have = sg == 0 ? Tch > 0 : true;
#pragma unroll
                        for (int g = 0; g < 4; ++g)
#pragma unroll
                            for (int e = 0; e < 16; e += 4) {
                                const int col = 16 * G[g] + e;
                                float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
                                if (have && (sg > 0 || col < R)) v = *reinterpret_cast<const float4*>(src + col);
                                av[g][e] = v.x; av[g][e + 1] = v.y; av[g][e + 2] = v.z; av[g][e + 3] = v.w;
                            }
#pragma unroll
                        for (int g = 0; g < 4; ++g) tc::tmem_st16(lane_addr + TM_AN + 16 * G[g], av[g]);
                        tc::tmem_wait_st();
                    }
                    // prefix B tile: rows 8 jj + 4 ch' + c  <-  span bhat tile jj, row 8 ch' + c
                    for (int i = ctid; i < len * 2 * C * 16; i += NCW * 32) {
                        const int j16 = i & 15, rowi = i >> 4;
                        const int c = rowi % C, c2 = (rowi / C) & 1, jj = rowi / (2 * C);
                        const int srow = 8 * c2 + c, drow = 8 * jj + 4 * c2 + c;
                        const int hv = j16 >> 3, jc = j16 & 7;
                        const uint4 v = *reinterpret_cast<const uint4*>(sm + OFF_SB + jj * 4096 + tc::sw128_chunk(16, hv, srow, jc));
                        *reinterpret_cast<uint4*>(sm + OFF_PB + tc::sw128_chunk(64, hv, drow, jc)) = v;
                    }
                    tc::fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) tc::mbar_arrive(&ctl->pbready);
                    const float a_anchor = s0 > 0 ? ac[s0 - 1] : 0.f;
                    for (int o = len - 1; o >= 0; --o) {
                        const int t = s0 + o;
                        const int buf = t & 1;
                        // ---- (1) prefix A rows for token t: L[t, s0+jj] xhat, and a zero pair row
                        if (npa >= 1) ok &= tc::mbar_wait(&ctl->pafree, ph_pafree.next(), abort);
                        ++npa;
                        {
                            // rows 8 jj + 4 ch' + c of the K-steps this token uses; a row holds
                            // L[t, s0+jj] xhat[ch', s0+jj, c, :] in column half ch' and zeros elsewhere
                            const int nrow_tok = (o % 2 == 0) ? o + 2 : o + 1;
                            for (int i = ctid; i < nrow_tok * 8 * 16; i += NCW * 32) {
                                const int j16 = i & 15, drow = i >> 4;
                                const int jj = drow >> 3, c2 = (drow >> 2) & 1, c = drow & 3;
                                const int hv = j16 >> 3, jc = j16 & 7;
                                uint4 w = make_uint4(0, 0, 0, 0);
                                if (hv == c2 && jj <= o && c < C) {
                                    const float* ac2 = acum + c2 * 64;
                                    const float L = __expf(ac2[t] - ac2[s0 + jj]);
                                    const uint4 v = *reinterpret_cast<const uint4*>(
                                        sm + OFF_SX + jj * 4096 + tc::sw128_chunk(16, c2, 8 * c2 + c, jc));
                                    w.x = tc::pack_bf16x2(L * bf16lo(v.x), L * bf16hi(v.x));
                                    w.y = tc::pack_bf16x2(L * bf16lo(v.y), L * bf16hi(v.y));
                                    w.z = tc::pack_bf16x2(L * bf16lo(v.z), L * bf16hi(v.z));
                                    w.w = tc::pack_bf16x2(L * bf16lo(v.w), L * bf16hi(v.w));
                                }
                                *reinterpret_cast<uint4*>(sm + OFF_PA + tc::sw128_chunk(64, hv, drow, jc)) = w;
                            }
                        }
                        tc::fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) tc::mbar_arrive(&ctl->pafull);
                        // cos / sin of this token's angles (both chunks), shared by all compute threads
                        const float* rawrot = reinterpret_cast<const float*>(sm + OFF_ROT + o * 1024);
                        float* coef = reinterpret_cast<float*>(sm + OFF_COEF + buf * 2048);
                        if (P.rot == ROT_PAIRWISE || P.rot == ROT_HALF) {
                            for (int i = ctid; i < 2 * P.na; i += NCW * 32) {
                                const int c2 = i / P.na, a = i - c2 * P.na;
                                float sv, cv;
                                sincosf(rawrot[c2 * 128 + a], &sv, &cv);
                                coef[c2 * 256 + a] = cv;
                                coef[c2 * 256 + 128 + a] = sv;
                            }
                        }
                        named_barrier_sync(1, NCW * 32);
                        // ---- (3) h_t from the prefix states and the anchor; d_da_{t+1}; c_t
                        ok &= tc::mbar_wait(&ctl->pfull, ph_pfull.next(), abort);
                        tc::tc_fence_after();
                        float h[4][16];
                        {
                            float an[4][16];
                            tmem_ld_row(lane_addr + TM_P, G, h);
                            tmem_ld_row(lane_addr + TM_AN, G, an);
                            tc::tc_fence_before();
                            __syncwarp();
                            if (lane == 0) tc::mbar_arrive(&ctl->pfree);
                            const float dsig = __expf(ac[t] - a_anchor);
#pragma unroll
                            for (int g = 0; g < 4; ++g)
#pragma unroll
                                for (int e = 0; e < 16; ++e) h[g][e] = fmaf(dsig, an[g][e], h[g][e]);
                        }
                        {
                            float dot = 0.f;
#pragma unroll
                            for (int g = 0; g < 4; ++g)
#pragma unroll
                                for (int e = 0; e < 16; ++e) dot = fmaf(gr[g][e], h[g][e], dot);
                            dot = warp_sum(dot);
                            if (lane == 0) atomicAdd(&rda[buf * 2 + ch], dot);
                        }
                        const bool live = t < Tch;
                        float c[4][16];
                        rotate_regs<false>(P, A.layoutB, G, h, coef + ch * 256, rawrot + ch * 128, c);
                        if (nc_ >= 1) ok &= tc::mbar_wait(&ctl->cfree, ph_cfree.next(), abort);
                        ++nc_;
                        write_tile_row(sm + OFF_C, m, G, c, !live);
                        tc::fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) tc::mbar_arrive(&ctl->cfull);
                        // ---- (5) d_c, d_rot, G, cotangent recurrence
                        ok &= tc::mbar_wait(&ctl->dcfull, ph_dcfull.next(), abort);
                        tc::tc_fence_after();
                        float dc[4][16];
                        tmem_ld_row(lane_addr + TM_DC, G, dc);
                        tc::tc_fence_before();
                        __syncwarp();
                        if (lane == 0) tc::mbar_arrive(&ctl->dcfree);
#pragma unroll
                        for (int g = 0; g < 4; ++g)
#pragma unroll
                            for (int e = 0; e < 16; ++e) dc[g][e] = live ? dc[g][e] + m1s[16 * G[g] + e] : 0.f;
                        // rotation-parameter gradient, reduced over the 64 rows of the chunk
                        if (P.rw) {
                            float cb[4][16];
                            read_tile_row(sm + OFF_C, m, G, cb);
                            float* rd = red + (buf * 2 + ch) * 128;
                            if (P.rot == ROT_QUAT) {
                                // sum_p d_c (x) conj(c) per block; d_Q = that (x) Q / |Q|^2 below
#pragma unroll
                                for (int part = 0; part < 2; ++part) {
                                    float v[32];
#pragma unroll
                                    for (int bq = 0; bq < 8; ++bq) {
                                        const int g = 2 * part + (bq >> 2), e = 4 * (bq & 3);
                                        float o0, o1, o2, o3;
                                        hamilton(dc[g][e], dc[g][e + 1], dc[g][e + 2], dc[g][e + 3], cb[g][e],
                                                 -cb[g][e + 1], -cb[g][e + 2], -cb[g][e + 3], o0, o1, o2, o3);
                                        v[4 * bq] = o0; v[4 * bq + 1] = o1; v[4 * bq + 2] = o2; v[4 * bq + 3] = o3;
                                    }
                                    transpose_reduce32(v, lane);
                                    const int bq = lane >> 2, g = 2 * part + (bq >> 2), e = 4 * (bq & 3);
                                    const int blk = (16 * G[g] + e) >> 2;
                                    if (blk < P.J) atomicAdd(&rd[4 * blk + (lane & 3)], v[0]);
                                }
                            } else if (P.rot == ROT_PAIRWISE) {
                                float v[32];
#pragma unroll
                                for (int g = 0; g < 4; ++g)
#pragma unroll
                                    for (int e = 0; e < 16; e += 2)
                                        v[8 * g + e / 2] = dc[g][e] * cb[g][e + 1] - dc[g][e + 1] * cb[g][e];
                                transpose_reduce32(v, lane);
                                const int g = lane >> 3, e = 2 * (lane & 7);
                                const int ang = (16 * G[g] + e) >> 1;
                                if (ang < P.na) atomicAdd(&rd[ang], v[0]);
                            } else {  // half-split: x columns in slots 0,1 (layout A) / slot 0 (layout B)
                                float v[32];
#pragma unroll
                                for (int e = 0; e < 16; ++e) {
                                    const int gb0 = A.layoutB ? 1 : 2;
                                    v[e] = dc[0][e] * cb[gb0][e] - dc[gb0][e] * cb[0][e];
                                    v[16 + e] = A.layoutB ? 0.f : (dc[1][e] * cb[3][e] - dc[3][e] * cb[1][e]);
                                }
                                transpose_reduce32(v, lane);
                                const int g = lane >> 4, e = lane & 15;
                                const int ang = 16 * G[g] + e;
                                if (!(A.layoutB && g == 1) && ang < P.na) atomicAdd(&rd[ang], v[0]);
                            }
                        }
                        {
                            float Gt[4][16];
                            rotate_regs<true>(P, A.layoutB, G, dc, coef + ch * 256, rawrot + ch * 128, Gt);
#pragma unroll
                            for (int g = 0; g < 4; ++g)
#pragma unroll
                                for (int e = 0; e < 16; ++e) gr[g][e] = fmaf(e_next, gr[g][e], Gt[g][e]);
                        }
                        const float e_t = e_of(t);
                        if (ng >= 1) ok &= tc::mbar_wait(&ctl->gfree, ph_gfree.next(), abort);
                        ++ng;
                        write_tile_row(sm + OFF_G, m, G, gr, false);
                        tc::fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) tc::mbar_arrive(&ctl->gfull);
                        named_barrier_sync(1, NCW * 32);
                        // ---- outputs of the reductions: d_rot_t and d_da_{t+1}
                        {
                            float* rd = red + buf * 256;
                            const int tot = 2 * 128;
                            for (int i = ctid; i < tot; i += NCW * 32) {
                                const int c2 = i >> 7, a = i & 127;
                                if (a < P.rw && I.exists[c2] && (2 * I.k + c2) < I.proc) {
                                    const int64_t o_r = off_rot(P, I.bb, (2 * I.k + c2) * FL + t, I.hh);
                                    float val = rd[i];
                                    if (P.rot == ROT_QUAT) {
                                        // (sum_p d_c (x) conj(c)) (x) Q / |Q|^2, component a & 3 of block a >> 2
                                        const float* raw = reinterpret_cast<const float*>(sm + OFF_ROT + o * 1024) + c2 * 128;
                                        const float* Q = raw + 4 * (a >> 2);
                                        const float s0q = rd[(i & ~3) + 0], s1q = rd[(i & ~3) + 1], s2q = rd[(i & ~3) + 2],
                                                    s3q = rd[(i & ~3) + 3];
                                        float o0, o1, o2, o3;
                                        hamilton(s0q, s1q, s2q, s3q, Q[0], Q[1], Q[2], Q[3], o0, o1, o2, o3);
                                        const float inv = 1.f / (Q[0] * Q[0] + Q[1] * Q[1] + Q[2] * Q[2] + Q[3] * Q[3]);
                                        const int comp = a & 3;
                                        val = inv * (comp == 0 ? o0 : comp == 1 ? o1 : comp == 2 ? o2 : o3);
                                    }
                                    B.drot[o_r + a] = val;
                                }
                            }
                            named_barrier_sync(1, NCW * 32);
                            for (int i = ctid; i < tot; i += NCW * 32) rd[i] = 0.f;
                            if (ctid < 2) {
                                const int c2 = ctid;
                                if (t + 1 < I.T[0] && I.exists[c2]) {
                                    const float e1 = __expf(ida[(c2 * 64 + t + 1) * 4 + (I.hh & 3)]);
                                    B.dda[off_da(P, I.bb, (2 * I.k + c2) * FL + t + 1, I.hh)] = e1 * rda[buf * 2 + c2];
                                }
                                rda[buf * 2 + c2] = 0.f;
                            }
                        }
                        e_next = e_t;
                        // ---- (7) d_xhat (lanes = rows) and d_bhat (lanes = r) of token t
                        ok &= tc::mbar_wait(&ctl->dxfull, ph_dxfull.next(), abort);
                        tc::tc_fence_after();
                        {
                            float v[8];
                            tc::tmem_ld8(lane_addr + TM_DX + 8 * ch, v);
                            float u[8];
                            tc::tmem_ld8(lane_addr + TM_DB + 8 * half, u);
                            tc::tmem_wait_ld();
                            tc::tc_fence_before();
                            __syncwarp();
                            if (lane == 0) tc::mbar_arrive(&ctl->dxfree);
                            if (half == 0 && chunk_ok) {
                                const int tok = n * FL + t;
#pragma unroll
                                for (int c = 0; c < 4; ++c)
                                    if (c < C) B.dx[off_x(P, I.bb, tok, c, I.hh) + pp] = __float2bfloat16_rn(v[c]);
                            }
                            if (m < R && I.exists[half]) {
                                const int tok = (2 * I.k + half) * FL + t;
#pragma unroll
                                for (int c = 0; c < 4; ++c)
                                    if (c < C) B.db[off_b(P, I.bb, tok, c, I.hh) + m] = __float2bfloat16_rn(u[c]);
                            }
                        }
                    }
                    __syncwarp();
                    if (lane == 0) tc::mbar_arrive(&ctl->spanfree);
                }
                // ---- chunk start: d_da_0 = e_0 <g_0, h_->, e_n = e_0 g_0 (anchor 0 = the carry)
                {
                    float an[4][16];
                    tmem_ld_row(lane_addr + TM_AN, G, an);
                    float dot = 0.f;
#pragma unroll
                    for (int g = 0; g < 4; ++g)
#pragma unroll
                        for (int e = 0; e < 16; ++e) dot = fmaf(gr[g][e], an[g][e], dot);
                    dot = warp_sum(dot);
                    if (lane == 0) atomicAdd(&rda[ch], dot);
                    named_barrier_sync(1, NCW * 32);
                    if (ctid < 2) {
                        const int c2 = ctid;
                        if (I.T[c2] > 0)
                            B.dda[off_da(P, I.bb, (2 * I.k + c2) * FL, I.hh)] =
                                __expf(ida[(c2 * 64) * 4 + (I.hh & 3)]) * rda[c2];
                        rda[c2] = 0.f;
                    }
                    if (Tch > 0) {
                        const float e0 = __expf(ida[(ch * 64) * 4 + (I.hh & 3)]);
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
            } else {
                // ================================ correction by the carry cotangent dH(n+1)
                const bool corr = chunk_ok && n + 1 < I.proc;
                float dh[4][16];
                {
                    const float* src = B.E + off_carry(P, I.bb, I.hh, n) + (int64_t)pp * R;
                    const float* hin = A.Hc + off_carry(P, I.bb, I.hh, n) + (int64_t)pp * R;
                    float dot = 0.f;
#pragma unroll
                    for (int g = 0; g < 4; ++g)
#pragma unroll
                        for (int e = 0; e < 16; e += 4) {
                            const int col = 16 * G[g] + e;
                            float4 v = make_float4(0.f, 0.f, 0.f, 0.f), hv = v;
                            if (corr && col < R) {
                                v = *reinterpret_cast<const float4*>(src + col);
                                hv = *reinterpret_cast<const float4*>(hin + col);
                            }
                            dh[g][e] = v.x; dh[g][e + 1] = v.y; dh[g][e + 2] = v.z; dh[g][e + 3] = v.w;
                            dot += v.x * hv.x + v.y * hv.y + v.z * hv.z + v.w * hv.w;
                        }
                    dot = warp_sum(dot);
                    if (lane == 0) atomicAdd(&rda[ch], dot);
                    if (ng >= 1) ok &= tc::mbar_wait(&ctl->gfree, ph_gfree.next(), abort);
                    ++ng;
                    write_tile_row(sm + OFF_G, m, G, dh, false);
                    tc::fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) tc::mbar_arrive(&ctl->gfull);
                }
                named_barrier_sync(1, NCW * 32);
                if (ctid < 2) {
                    base[ctid] = __expf(acum[ctid * 64 + 63]) * rda[ctid];
                    rda[ctid] = 0.f;
                }
                const float alast = ac[63];
                const bool corr_b = I.exists[half] && (2 * I.k + half) + 1 < I.proc;
                const float alast_b = acum[half * 64 + 63];
                for (int t = 0; t < I.T[0]; ++t, ++q) {
                    const uint32_t s = q % NS;
                    ok &= tc::mbar_wait(&ctl->full[s], ph_full[s].next(), abort);
                    ok &= tc::mbar_wait(&ctl->dxfull, ph_dxfull.next(), abort);
                    tc::tc_fence_after();
                    float v[8], u[8];
                    tc::tmem_ld8(lane_addr + TM_DX + 8 * ch, v);
                    tc::tmem_ld8(lane_addr + TM_DB + 8 * half, u);
                    tc::tmem_wait_ld();
                    tc::tc_fence_before();
                    __syncwarp();
                    if (lane == 0) tc::mbar_arrive(&ctl->dxfree);
                    // omega_t = sum_c <xhat_tc, U_tc> over this chunk's rows (U = dH bhat^T)
                    float w = 0.f;
                    if (half == 0) {
                        const unsigned char* xt = sm + OFF_RING + s * 8192;
#pragma unroll
                        for (int c = 0; c < 4; ++c)
                            if (c < C) {
                                const uint32_t off = tc::sw128_offset(16, 8 * ch + c, 64 * ch + pp);
                                const float xv = __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(xt + off));
                                w = fmaf(xv, v[c], w);
                            }
                    }
                    w = warp_sum(w);
                    __syncwarp();
                    if (lane == 0) {
                        tc::mbar_arrive(&ctl->empty[s]);
                        if (half == 0) atomicAdd(&om[ch * 64 + t], w);
                    }
                    if (half == 0 && corr) {
                        const float sc = __expf(alast - ac[t]);
                        const int tok = n * FL + t;
#pragma unroll
                        for (int c = 0; c < 4; ++c)
                            if (c < C) {
                                __nv_bfloat16* d = B.dx + off_x(P, I.bb, tok, c, I.hh) + pp;
                                *d = __float2bfloat16_rn(__bfloat162float(*d) + sc * v[c]);
                            }
                    }
                    if (m < R && corr_b) {
                        const float sc = __expf(alast_b - acum[half * 64 + t]);
                        const int tok = (2 * I.k + half) * FL + t;
#pragma unroll
                        for (int c = 0; c < 4; ++c)
                            if (c < C) {
                                __nv_bfloat16* d = B.db + off_b(P, I.bb, tok, c, I.hh) + m;
                                *d = __float2bfloat16_rn(__bfloat162float(*d) + sc * u[c]);
                            }
                    }
                }
                named_barrier_sync(1, NCW * 32);
                // d_da_s += D_n <dH, h_-> + sum_{j<s} sc_j omega_j
                if (ctid < 128) {
                    const int c2 = ctid >> 6, s = ctid & 63;
                    const int n2 = 2 * I.k + c2;
                    if (I.exists[c2] && n2 + 1 < I.proc) {
                        const float* ac2 = acum + c2 * 64;
                        float pre = 0.f;
                        for (int j = 0; j < s; ++j) pre += __expf(ac2[63] - ac2[j]) * om[c2 * 64 + j];
                        B.dda[off_da(P, I.bb, n2 * FL + s, I.hh)] += base[c2] + pre;
                    }
                }
                named_barrier_sync(1, NCW * 32);
                if (ctid < 128) om[ctid] = 0.f;
            }
            if (MODE == LOCAL) {
                // the forward-sweep ring shares memory with the prefix tiles: restore the zero
                // padding rows the next item's W products rely on
                for (uint32_t i = ctid; i < 32768 / 16; i += NCW * 32)
                    reinterpret_cast<uint4*>(sm + OFF_RING)[i] = make_uint4(0, 0, 0, 0);
                tc::fence_proxy_async_smem();
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

}  // namespace fastbwd

// ----------------------------------------------------------------------------- host side
namespace fastk {

size_t bwd_anchor_bytes() { return (size_t)kMaxBwdGrid * fastbwd::NANCHOR * 128 * 128 * sizeof(float); }

cudaError_t launch_tc_bwd(int mode, const FastArgs& fa, float* E, float* anchors, const float* dm2, const float* dm1,
                          void* dx, void* db, float* dda, float* drot, const TensorMaps& maps, int grid,
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
    auto kern = mode == LOCAL ? tc_bwd_kernel<LOCAL> : tc_bwd_kernel<CORR>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BYTES);
    if (e != cudaSuccess) return e;
    const int kid = mode == LOCAL ? KID_FAST_BWD : KID_FAST_CORRECT;
    mm_prof_mark(kid, 1, st);
    kern<<<grid, NTHR, SMEM_BYTES, st>>>(a, maps.x, maps.b, maps.rot, maps.da64);
    mm_prof_mark(kid, 0, st);
    return cudaGetLastError();
}

}  // namespace fastk
