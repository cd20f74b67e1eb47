// fast_fwd.cu -- tcgen05 / TMA forward of the state-moments operator (bf16 operands, 64 state
// rows per head -- larger p as 64-row groups run as heads --, r up to 128, C <= 8).
//
// One persistent CTA per SM walks a contiguous range of work items; an item is a pair of
// 64-token chunks of one (batch row, head).  The two chunks share the 128 TMEM lanes:
// row m = (chunk ch, per-head index p), so every per-token quantity is a 128 x r tile.
//
//   warp 8 (TMA)    : per token, xhat/bhat rows of both chunks (128-byte swizzle), the
//                     token's rotation parameters and da, into a 4-stage ring; the copies of a
//                     token are issued from different lanes.
//   warp 9 (MMA)    : W_t = sum_c xhat_tc (x) bhat_tc for both chunks as ONE block-diagonal
//                     MMA (M = 128 rows, N = 128, K = 16 = (chunk, channel) rows), into one of
//                     two TMEM accumulators; then the moment MMAs m2 += c^T [c | 1] over the
//                     128 rows (8 x K=16 steps, N = 144: column 128 of the ones block gives m1).
//   warps 0-7       : two threads per row (64 columns each, two 32-column passes whose rotation
//                     partners stay inside the pass).  h = e^{da} h + W in fp32 registers (the
//                     chunk recurrence h~[t] = d_t h_- + sum_j L[t,j] W_j unrolled), de-rotation
//                     in registers, masking, bf16 c rows into the swizzled smem tile that both
//                     moment operands read.
//
// The cos / sin of a token's angles are evaluated per warp (one angle per lane, the ones this
// warp's columns need) into a small per-warp table, so that no block-wide barrier is needed per
// token.  The chunk-entry carries come from the chunk-end states (fast_end.cu) and the carry scan.
//
// Every wait is bounded; a wait that gives up sets the workspace error word and the CTA winds
// down (compute warps keep stepping through their loops so named barriers stay matched).
#include <cuda.h>

#include "common.cuh"
#include "fast.h"
#include "fast_common.cuh"
#include "prof.h"
#include "rot_sincos.cuh"
#include "tc.cuh"

namespace fastfwd {

using namespace fastk;

constexpr int NTHR = 320;
constexpr int WARP_TMA = 8, WARP_MMA = 9;
constexpr int NS = 4;  // staging ring depth

// shared memory map (bytes from a 1024-aligned base)
constexpr uint32_t C_BYTES = 49152;                    // c tile: 2 x 16 KB halves + 16 KB ones block
constexpr uint32_t OFF_C = 0;                          // 2 c tiles
constexpr uint32_t OFF_X = 2 * C_BYTES;                // NS x 4 KB  (16 K-rows x 128 (ch,p))
constexpr uint32_t OFF_B = OFF_X + NS * 4096;          // NS x 4 KB  (16 K-rows x 128 r)
constexpr uint32_t OFF_ROT = OFF_B + NS * 4096;        // NS x 2 chunks x 512 B raw rotation
constexpr uint32_t OFF_DA = OFF_ROT + NS * 1024;       // NS x 2 chunks x 128 B slots (4 heads of da)
constexpr uint32_t OFF_TBL = OFF_DA + NS * 256;        // 8 warps x (32 cos | 32 sin) fp32
constexpr uint32_t OFF_CTL = OFF_TBL + NCW * 64 * 4;
constexpr uint32_t SMEM_BYTES = OFF_CTL + 256 + 1024;

struct Ctl {
    uint64_t full[NS], empty[NS];
    uint64_t wfull[2], wfree[2];
    uint64_t cfull[2], cfree[2];
    uint64_t segdone, segfree, fin;
    uint32_t tbase;
    int abort;
};
static_assert(sizeof(Ctl) <= 256, "control block");
// tensor copies need 128-byte aligned shared destinations (1024 for the swizzled tiles)
static_assert(OFF_X % 1024 == 0 && OFF_B % 1024 == 0 && OFF_C % 1024 == 0, "swizzled tiles");
static_assert(OFF_ROT % 128 == 0 && OFF_DA % 128 == 0 && OFF_CTL % 8 == 0, "tensor-copy slots");

constexpr uint32_t TM_W = 0, TM_M2 = 256, TM_COLS = 512;

__device__ __forceinline__ void fail(Ctl* ctl, int* err, int code) {
    ctl->abort = 1;
    atomicExch(err, code);
}

// DAT: da comes by 4-head tensor copies (h a multiple of 4), else by plain loads of the one head
template <int ROTK, int LAYB, bool DAT>
__global__ void __launch_bounds__(NTHR, 1)
    tc_fwd_kernel(const __grid_constant__ FastArgs A, const __grid_constant__ CUtensorMap tmx,
                  const __grid_constant__ CUtensorMap tmb, const __grid_constant__ CUtensorMap tmr,
                  const __grid_constant__ CUtensorMap tmd) {
    extern __shared__ unsigned char smraw[];
    unsigned char* sm = smraw + ((1024u - (tc::smem_u32(smraw) & 1023u)) & 1023u);
    Ctl* ctl = reinterpret_cast<Ctl*>(sm + OFF_CTL);
    const MMParams& P = A.P;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int R = P.r;

    // ---- work range of this CTA
    const int it0 = item_begin(A, blockIdx.x), it1 = item_begin(A, blockIdx.x + 1);

    // ---- one-time set-up: zero the staged operand tiles, the ones block, barriers, TMEM
    for (uint32_t i = tid; i < (OFF_ROT - OFF_X) / 16; i += NTHR)
        reinterpret_cast<uint4*>(sm + OFF_X)[i] = make_uint4(0, 0, 0, 0);
    {
        // ones block of both c tiles: column 128 (first column of the block) = 1.0, rest 0
        for (uint32_t i = tid; i < 2 * 128; i += NTHR) {
            const uint32_t buf = i >> 7, row = i & 127;
            unsigned char* base = sm + OFF_C + buf * C_BYTES + 32768;
            for (uint32_t j = 0; j < 8; ++j) {
                uint4 v = make_uint4(0, 0, 0, 0);
                if (j == 0) v.x = 0x3F80u;  // bf16(1.0) in the low half of the first word
                *reinterpret_cast<uint4*>(base + tc::sw128_chunk(128, 0, row, j)) = v;
            }
        }
    }
    if (tid == 0) {
        for (int s = 0; s < NS; ++s) {
            tc::mbar_init(&ctl->full[s], 1);
            tc::mbar_init(&ctl->empty[s], 1 + NCW);
        }
        for (int i = 0; i < 2; ++i) {
            tc::mbar_init(&ctl->wfull[i], 1);
            tc::mbar_init(&ctl->wfree[i], NCW);
            tc::mbar_init(&ctl->cfull[i], NCW);
            tc::mbar_init(&ctl->cfree[i], 1);
        }
        tc::mbar_init(&ctl->segdone, 1);
        tc::mbar_init(&ctl->segfree, NCW);
        tc::mbar_init(&ctl->fin, 1);
        ctl->abort = 0;
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

    if (warp == WARP_TMA) {
        // ================================================================ TMA producer
        // The whole warp runs the loop: lane 0 arms the stage barrier and the copies of a token
        // (xhat rows, bhat column blocks, rotation row and da of both chunks) go out from
        // different lanes, since one copy issue costs a thread about 100 cycles.  Wait results are
        // made warp-uniform so that all lanes leave together.
        uint32_t q = 0;
        bool ok = true;
        const int nbx = 1 + (R + 63) / 64, ncp = nbx + (P.rw ? 1 : 0) + 1;  // copies per token and chunk
        for (int it = it0; it < it1 && ok; ++it) {
            const Item I = decode_item(A, it);
            for (int t = 0; t < I.T[0] && ok; ++t, ++q) {
                const uint32_t s = q % NS, u = q / NS;
                if (u >= 1) ok = __all_sync(0xffffffffu, tc::mbar_wait(&ctl->empty[s], (u - 1) & 1, abort));
                if (!ok) break;
                if (!DAT) {
                    // this head's da of the token, into the slot position the 4-head copy would fill,
                    // stored before the arrival that publishes the stage
                    if (lane < 2 && t < I.T[lane]) {  // (no read past the row's end)
                        const int row = I.bb * P.s + (2 * I.k + lane) * FL + t;
                        reinterpret_cast<float*>(sm + OFF_DA + s * 256 + lane * 128)[I.hd & 3] =
                            A.da[(int64_t)row * P.heads + I.hd];
                    }
                    __syncwarp();
                }
                if (lane == 0) {
                    uint32_t bytes = 0;
                    for (int ch = 0; ch < 2; ++ch)
                        if (I.exists[ch]) bytes += stage_bytes(A);
                    tc::mbar_arrive_expect_tx(&ctl->full[s], bytes);
                }
                __syncwarp();
                if (lane < 2 * ncp) {
                    const int ch = lane >= ncp ? 1 : 0, kind = lane - ch * ncp;
                    if (ch ? I.exists[1] : I.exists[0]) {
                        const int row = I.bb * P.s + (2 * I.k + ch) * FL + t;
                        if (kind == 0)
                            tc::tma_load_4d(sm + OFF_X + s * 4096 + ch * 3072, &tmx, 0, I.hh, 0, row, &ctl->full[s]);
                        else if (kind < nbx)
                            tc::tma_load_4d(sm + OFF_B + s * 4096 + (kind - 1) * 2048 + ch * 1024, &tmb, 64 * (kind - 1),
                                            I.hd, 0, row, &ctl->full[s]);
                        else if (P.rw && kind == nbx)
                            tc::tma_load_3d(sm + OFF_ROT + s * 1024 + ch * 512, &tmr, 0, I.hd, row, &ctl->full[s]);
                        else if (DAT)
                            tc::tma_load_2d(sm + OFF_DA + s * 256 + ch * 128, &tmd, I.hd & ~3, row, &ctl->full[s]);
                    }
                }
            }
        }
        if (lane == 0) {
            if (!ok) fail(ctl, A.err, 11);
            // drain: every issued stage must land before the CTA exits (own bounded wait,
            // independent of the abort flag)
            int never = 0;
            for (uint32_t s = 0; s < NS && q > s; ++s) {
                const uint32_t last = (q - 1 - s) / NS;  // last use index of stage s
                tc::mbar_wait(&ctl->full[s], last & 1, &never, 1u << 20);
            }
        }
    } else if (warp == WARP_MMA) {
        // ================================================================ MMA issuer
        if (lane == 0) {
            const uint32_t idW = tc::idesc_bf16(128, 128, 1, 1);
            const uint32_t idM = tc::idesc_bf16(128, 144, 1, 1);
            const uint32_t xs0 = tc::smem_u32(sm + OFF_X), bs0 = tc::smem_u32(sm + OFF_B);
            const uint32_t cs0 = tc::smem_u32(sm + OFF_C);
            TokenWalk walk(A, it0, it1);
            // W for flat token qq: stage qq % NS, accumulator qq % 2
            auto issue_w = [&](uint32_t qq) -> bool {
                const uint32_t s = qq % NS, u = qq / NS, wb = qq & 1, uw = qq >> 1;
                if (!tc::mbar_wait(&ctl->full[s], u & 1, abort)) return false;
                if (uw >= 1 && !tc::mbar_wait(&ctl->wfree[wb], (uw - 1) & 1, abort)) return false;
                tc::tc_fence_after();
                const uint64_t ad = tc::sdesc_sw128(xs0 + s * 4096, 2048, 1024);
                const uint64_t bd = tc::sdesc_sw128(bs0 + s * 4096, 2048, 1024);
                tc::mma_bf16(tbase + TM_W + wb * 128, ad, bd, idW, 0);
                tc::mma_commit(&ctl->wfull[wb]);
                tc::mma_commit(&ctl->empty[s]);
                return true;
            };
            const uint32_t ntok = walk.total_tokens();
            bool ok = ntok == 0 || issue_w(0);
            uint32_t seg = 0;
            for (uint32_t q = 0; ok && q < ntok; ++q) {
                const TokenInfo ti = walk.next();
                if (q + 1 < ntok && !issue_w(q + 1)) { ok = false; break; }
                {
                    const uint32_t cb = q & 1, uc = q >> 1;
                    if (!tc::mbar_wait(&ctl->cfull[cb], uc & 1, abort)) { ok = false; break; }
                    if (ti.seg_first && seg >= 1 && !tc::mbar_wait(&ctl->segfree, (seg - 1) & 1, abort)) {
                        ok = false;
                        break;
                    }
                    tc::tc_fence_after();
                    const uint32_t cbase = cs0 + cb * C_BYTES;
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks) {
                        const uint64_t d = tc::sdesc_sw128(cbase + ks * 2048, 16384, 1024);
                        tc::mma_bf16(tbase + TM_M2, d, d, idM, (ti.seg_first && ks == 0) ? 0u : 1u);
                    }
                    tc::mma_commit(&ctl->cfree[cb]);
                    if (ti.seg_last) {
                        tc::mma_commit(&ctl->segdone);
                        ++seg;
                    }
                }
            }
            if (!ok) fail(ctl, A.err, 12);
            tc::mma_commit(&ctl->fin);
            int never = 0;  // in-flight MMAs must finish before the TMEM is released
            tc::mbar_wait(&ctl->fin, 0, &never, 1u << 20);
        }
    } else {
        // ================================================================ compute warps
        const int half = warp >> 2;              // which 64 columns of the row
        const int m = ((warp & 3) << 5) + lane;  // TMEM lane = row (chunk, p)
        const int ch = m >> 6, pp = m & 63;
        int G[4];
        col_groups(LAYB, half, G);
        const uint32_t lane_addr = tbase + ((uint32_t)((warp & 3) * 32) << 16);
        float* tbl = reinterpret_cast<float*>(sm + OFF_TBL) + warp * 64;  // this warp's cos | sin
        // the angle this lane evaluates for the warp's table (table slot = lane)
        int my_ang = 1 << 30;
        if (ROTK == ROT_PAIRWISE) {  // slot g pair i  <->  table 8 g + i
            const int g = lane >> 3;
            my_ang = 8 * (g == 0 ? G[0] : g == 1 ? G[1] : g == 2 ? G[2] : G[3]) + (lane & 7);
        } else if (ROTK == ROT_HALF) {  // pass p element e  <->  table 16 p + e
            if (!LAYB) my_ang = 16 * (lane < 16 ? G[0] : G[1]) + (lane & 15);
            else if (lane < 16) my_ang = 16 * G[0] + lane;
        }
        float S[4][16];
        uint32_t q = 0, seg = 0;
        int seg_k0 = 0, seg_it0 = it0;  // pair index and item of the current segment's first item
        bool ok = true;
        auto check = [&](bool r) {  // the first failed wait stops the whole CTA at once
            if (!r && ok) {
                ok = false;
                fail(ctl, A.err, 13);
            }
        };
        for (int it = it0; it < it1; ++it) {
            const Item I = decode_item(A, it);
            const int Tch = ch ? I.T[1] : I.T[0];
            const int n = 2 * I.k + ch;
            if (I.seg_first) {
                seg_k0 = I.k;
                seg_it0 = it;
            }
            // chunk-entry carry
            if (Tch > 0) {
                const float* src = A.Hc + off_carry(P, I.bb, I.hh, n) + (int64_t)pp * R;
#pragma unroll
                for (int g = 0; g < 4; ++g)
#pragma unroll
                    for (int e = 0; e < 16; e += 4) {
                        const int col = 16 * G[g] + e;
                        const float4 v =
                            col < R ? *reinterpret_cast<const float4*>(src + col) : make_float4(0.f, 0.f, 0.f, 0.f);
                        S[g][e] = v.x; S[g][e + 1] = v.y; S[g][e + 2] = v.z; S[g][e + 3] = v.w;
                    }
            } else {
#pragma unroll
                for (int g = 0; g < 4; ++g)
#pragma unroll
                    for (int e = 0; e < 16; ++e) S[g][e] = 0.f;
            }
            for (int t = 0; t < I.T[0]; ++t, ++q) {
                const uint32_t s = q % NS, u = q / NS;
                check(tc::mbar_wait(&ctl->full[s], u & 1, abort));
                const bool live = t < Tch;
                if (t == Tch) {  // the chunk's valid tokens are done: from here its c rows are zero
#pragma unroll
                    for (int g = 0; g < 4; ++g)
#pragma unroll
                        for (int e = 0; e < 16; ++e) S[g][e] = 0.f;
                }
                const float et = live ? __expf(reinterpret_cast<const float*>(sm + OFF_DA + s * 256 + ch * 128)[I.hd & 3])
                                      : 1.f;
                const float* qt = reinterpret_cast<const float*>(sm + OFF_ROT + s * 1024 + ch * 512);
                if (ROTK == ROT_PAIRWISE || ROTK == ROT_HALF) {
                    float sv = 0.f, cv = 1.f;
                    if (my_ang < P.na) rot_sincos(qt[my_ang], &sv, &cv);
                    __syncwarp();  // the previous token's table has been read
                    tbl[lane] = cv;
                    tbl[32 + lane] = sv;
                    __syncwarp();
                }
                const uint32_t wb = q & 1, uw = q >> 1, cb = q & 1, uc = q >> 1;
                check(tc::mbar_wait(&ctl->wfull[wb], uw & 1, abort));
                if (uc >= 1) check(tc::mbar_wait(&ctl->cfree[cb], (uc - 1) & 1, abort));
                tc::tc_fence_after();
                unsigned char* ct = sm + OFF_C + cb * C_BYTES;
                // all four column groups of W_t in one tensor-memory round trip
                float Wt[4][16];
#pragma unroll
                for (int g = 0; g < 4; ++g) tc::tmem_ld16(lane_addr + TM_W + wb * 128 + 16 * G[g], Wt[g]);
                tc::tmem_wait_ld();
                tc::tc_fence_before();
                __syncwarp();
                if (lane == 0) tc::mbar_arrive(&ctl->wfree[wb]);
#pragma unroll
                for (int pass = 0; pass < 2; ++pass) {
                    const int sa = slot_a<LAYB>(pass), sb = slot_b<LAYB>(pass);
                    float(&a)[16] = Wt[sa];
                    float(&b)[16] = Wt[sb];
                    if (live) {
#pragma unroll
                        for (int e = 0; e < 16; e += 2) {
                            ffma2(S[sa][e], S[sa][e + 1], et, et, S[sa][e], S[sa][e + 1], a[e], a[e + 1]);
                            ffma2(S[sb][e], S[sb][e + 1], et, et, S[sb][e], S[sb][e + 1], b[e], b[e + 1]);
                        }
                    }
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        a[e] = S[sa][e];
                        b[e] = S[sb][e];
                    }
                    // de-rotation c = R_t h of the pass's two slots
                    if (ROTK == ROT_PAIRWISE) {
#pragma unroll
                        for (int sl = 0; sl < 2; ++sl) {
                            if (!group_rotated<ROTK>(P, G[sl ? sb : sa])) continue;  // identity
                            float(&v)[16] = sl ? b : a;
                            const int ti = 8 * (sl ? sb : sa);
                            float cs[8], sn[8];
                            *reinterpret_cast<float4*>(&cs[0]) = *reinterpret_cast<const float4*>(tbl + ti);
                            *reinterpret_cast<float4*>(&cs[4]) = *reinterpret_cast<const float4*>(tbl + ti + 4);
                            *reinterpret_cast<float4*>(&sn[0]) = *reinterpret_cast<const float4*>(tbl + 32 + ti);
                            *reinterpret_cast<float4*>(&sn[4]) = *reinterpret_cast<const float4*>(tbl + 36 + ti);
#pragma unroll
                            for (int e = 0; e < 16; e += 2) {
                                const float x = v[e], y = v[e + 1];
                                v[e] = fmaf(cs[e / 2], x, sn[e / 2] * y);
                                v[e + 1] = fmaf(cs[e / 2], y, -sn[e / 2] * x);
                            }
                        }
                    } else if (ROTK == ROT_HALF) {
                        if (!(LAYB && pass == 1) && group_rotated<ROTK>(P, G[sa])) {
                            const int ti = 16 * pass;
#pragma unroll
                            for (int e4 = 0; e4 < 16; e4 += 4) {
                                const float4 c4 = *reinterpret_cast<const float4*>(tbl + ti + e4);
                                const float4 s4 = *reinterpret_cast<const float4*>(tbl + 32 + ti + e4);
                                const float cs[4] = {c4.x, c4.y, c4.z, c4.w}, sn[4] = {s4.x, s4.y, s4.z, s4.w};
#pragma unroll
                                for (int j = 0; j < 4; j += 2) {
                                    const int e = e4 + j;
                                    const float x0 = a[e], x1 = a[e + 1], y0 = b[e], y1 = b[e + 1];
                                    float u0, u1, w0, w1;
                                    fmul2(u0, u1, sn[j], sn[j + 1], y0, y1);    // s y
                                    fmul2(w0, w1, -sn[j], -sn[j + 1], x0, x1);  // -s x
                                    ffma2(a[e], a[e + 1], cs[j], cs[j + 1], x0, x1, u0, u1);
                                    ffma2(b[e], b[e + 1], cs[j], cs[j + 1], y0, y1, w0, w1);
                                }
                            }
                        }
                    } else if (ROTK == ROT_QUAT) {
#pragma unroll
                        for (int sl = 0; sl < 2; ++sl) {
                            if (!group_rotated<ROTK>(P, G[sl ? sb : sa])) continue;  // identity
                            float(&v)[16] = sl ? b : a;
                            const int k0 = 16 * G[sl ? sb : sa];
#pragma unroll
                            for (int e = 0; e < 16; e += 4) {
                                const int blk = (k0 + e) >> 2;
                                if (blk < P.J) {
                                    const float* Q = qt + 4 * blk;
                                    hamilton(Q[0], Q[1], Q[2], Q[3], v[e], v[e + 1], v[e + 2], v[e + 3], v[e], v[e + 1],
                                             v[e + 2], v[e + 3]);
                                }
                            }
                        }
                    }
                    // (past the chunk's valid tokens S is zero, and so is its de-rotation)
                    write_tile16(ct, m, G[sa], a, false);
                    write_tile16(ct, m, G[sb], b, false);
                }
                tc::fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    tc::mbar_arrive(&ctl->cfull[cb]);
                    tc::mbar_arrive(&ctl->empty[s]);
                }
            }
            if (I.seg_last) {
                // flush the (b,h) moment accumulator (lanes are rows r1 of m2) with plain stores:
                // into m2 / m1 when this segment covers every chunk pair of (b,h), else into this
                // CTA's partial slot (0 for its first segment, 1 for its last), which the reduce
                // kernel sums in CTA order, so that the result does not depend on timing
                check(tc::mbar_wait(&ctl->segdone, seg & 1, abort));
                tc::tc_fence_after();
                const bool whole = seg_k0 == 0 && I.k == pairs_of(P, I.bb) - 1;
                // the item's head again (the token steps use only the caller's head, I.hd)
                int fb, fh, fk;
                locate(A, it, fb, fh, fk);
                float* M2 = whole ? A.m2 + ((int64_t)fb * P.h + fh) * P.r * P.r
                                  : A.m2p + (int64_t)(2 * blockIdx.x + (seg_it0 == it0 ? 0 : 1)) * (P.r * P.r + P.r);
                float* M1 = whole ? A.m1 + ((int64_t)fb * P.h + fh) * P.r : M2 + P.r * P.r;
#pragma unroll
                for (int g = 0; g < 4; ++g) {
                    float v[16];
                    const int c0 = 64 * half + 16 * g;
                    tc::tmem_ld16(lane_addr + TM_M2 + c0, v);
                    tc::tmem_wait_ld();
                    if (m < R && c0 < R) {
                        float4* dst = reinterpret_cast<float4*>(M2 + (int64_t)m * P.r + c0);
#pragma unroll
                        for (int e = 0; e < 16; e += 4) dst[e / 4] = make_float4(v[e], v[e + 1], v[e + 2], v[e + 3]);
                    }
                }
                if (half == 0) {
                    float v[8];
                    tc::tmem_ld8(lane_addr + TM_M2 + 128, v);
                    tc::tmem_wait_ld();
                    if (m < R) M1[m] = v[0];
                }
                tc::tc_fence_before();
                __syncwarp();
                if (lane == 0) tc::mbar_arrive(&ctl->segfree);
                ++seg;
            }
        }
    }
    // ---- teardown
    tc::tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc::tc_fence_after();
        tc::tmem_dealloc(tbase, TM_COLS);
    }
}

// Moments of the (b,h) pairs whose chunk pairs were split over several CTAs: the partial slots
// of the CTAs that worked on them, summed in CTA order.  Grid x is the (b,h), grid y a slice of
// its r r + r moments; pairs done by one CTA were stored by it directly.
__global__ void __launch_bounds__(256) k_m2_reduce(const __grid_constant__ FastArgs A, int grid) {
    const MMParams& P = A.P;
    __shared__ int slots[kMaxFwdGrid];
    __shared__ int nslots;
    const int bb = blockIdx.x / P.h, hh = blockIdx.x - bb * P.h;
    if (threadIdx.x == 0) {
        int i0 = 0;
        for (int b2 = 0; b2 < bb; ++b2) i0 += P.h * pairs_of(P, b2);
        const int np = pairs_of(P, bb);
        int n = 0;
        if (np > 0) {
            i0 += hh * np;
            const int i1 = i0 + np;  // items [i0, i1) of (bb, hh)
            // the CTAs whose ranges meet [i0, i1), in order: CTA c holds [begin(c), begin(c+1));
            // start from an estimate of the CTA holding i0 and step to it
            int c = (int)(((int64_t)i0 * grid) / A.items);
            while (c + 1 < grid && item_begin_of(A.items, grid, c + 1) <= i0) ++c;
            while (c > 0 && item_begin_of(A.items, grid, c) > i0) --c;
            for (; c < grid && item_begin_of(A.items, grid, c) < i1 && n < kMaxFwdGrid; ++c) {
                const int c_lo = item_begin_of(A.items, grid, c);
                slots[n++] = 2 * c + (c_lo >= i0 ? 0 : 1);
            }
        }
        nslots = n < 2 ? 0 : n;  // one CTA: it stored the pair itself
    }
    __syncthreads();
    const int ns = nslots;
    if (ns == 0) return;
    const int nel4 = (P.r * P.r + P.r) / 4;  // r is a multiple of 4: whole float4 pieces
    // blockIdx.y picks a slice of blockDim.x float4 pieces: one piece per thread, its slot loads
    // all independent, so the short reduction is not latency-bound on a few blocks
    const int e = blockIdx.y * blockDim.x + threadIdx.x;
    if (e >= nel4) return;
    float4* M2 = reinterpret_cast<float4*>(A.m2 + ((int64_t)bb * P.h + hh) * P.r * P.r);
    float4* M1 = reinterpret_cast<float4*>(A.m1 + ((int64_t)bb * P.h + hh) * P.r);
    const float4* src = reinterpret_cast<const float4*>(A.m2p);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
    for (int i = 0; i < ns; ++i) {
        const float4 v = src[(int64_t)slots[i] * nel4 + e];
        acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
    }
    if (4 * e < P.r * P.r) M2[e] = acc;
    else M1[e - P.r * P.r / 4] = acc;
}

}  // namespace fastfwd

// ----------------------------------------------------------------------------- host side
namespace fastk {

cudaError_t launch_tc_fwd(const FastArgs& args, const TensorMaps& maps, int grid, cudaStream_t st) {
    using namespace fastfwd;
    decltype(&tc_fwd_kernel<ROT_NONE, 0, true>) kern;
    const bool dat = da_by_tma(args.P);
    switch (args.P.rot) {
        case ROT_PAIRWISE: kern = dat ? tc_fwd_kernel<ROT_PAIRWISE, 0, true> : tc_fwd_kernel<ROT_PAIRWISE, 0, false>; break;
        case ROT_HALF:
            kern = args.layoutB ? (dat ? tc_fwd_kernel<ROT_HALF, 1, true> : tc_fwd_kernel<ROT_HALF, 1, false>)
                                : (dat ? tc_fwd_kernel<ROT_HALF, 0, true> : tc_fwd_kernel<ROT_HALF, 0, false>);
            break;
        case ROT_QUAT: kern = dat ? tc_fwd_kernel<ROT_QUAT, 0, true> : tc_fwd_kernel<ROT_QUAT, 0, false>; break;
        default: kern = dat ? tc_fwd_kernel<ROT_NONE, 0, true> : tc_fwd_kernel<ROT_NONE, 0, false>; break;
    }
    cudaError_t e = mm_allow_smem(reinterpret_cast<const void*>(kern), (int)SMEM_BYTES);
    if (e != cudaSuccess) return e;
    mm_prof_mark(KID_FAST_FWD, 1, st);
    kern<<<grid, NTHR, SMEM_BYTES, st>>>(args, maps.x, maps.b, maps.rot, maps.da);
    mm_prof_mark(KID_FAST_FWD, 0, st);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if (grid == 1) return cudaSuccess;  // one CTA stored every (b,h) itself
    mm_prof_mark(KID_M2_REDUCE, 1, st);
    const int nel4 = (args.P.r * args.P.r + args.P.r) / 4;
    k_m2_reduce<<<dim3(args.P.b * args.P.h, (nel4 + 255) / 256), 256, 0, st>>>(args, grid);
    mm_prof_mark(KID_M2_REDUCE, 0, st);
    return cudaGetLastError();
}

size_t fwd_partial_bytes(const MMParams& P) {
    // the grid never exceeds the work items, whose number is at most b h ceil(nc / 2)
    const int64_t items = (int64_t)P.b * P.h * ((P.nc + 1) / 2);
    const int64_t grid = items < kMaxFwdGrid ? items : kMaxFwdGrid;
    return (size_t)(2 * grid) * ((size_t)P.r * P.r + P.r) * sizeof(float);
}

}  // namespace fastk
