// fast_corr.cu -- boundary-cotangent correction of the recompute backward as two GEMMs per chunk.
//
// For every chunk n but the last processed one, with dH = dH(n+1) the cotangent of the state the
// chunk hands on ("mamba3/moments/backward.rs", module header "Gradient math": the d_h+ terms),
// sc_t = exp(a_last - a_t) and a_t the inclusive cumulative sum of da inside the chunk:
//
//   U_{t,c} = dH bhat_{t,c}   (p values)          d_xhat_{t,c} += sc_t U_{t,c}
//   V_{t,c} = dH^T xhat_{t,c} (r values)          d_bhat_{t,c} += sc_t V_{t,c}
//   omega_t = sum_c <xhat_{t,c}, U_{t,c}>          d_da_s += D_n <dH, h_-(n)> + sum_{j<s} sc_j omega_j
//
// Over the rows (t, c) of a stage of TPS tokens (32, or 16 when C > 4) these are U = Bhat dH^T
// (M = TPS C <= 128, N = p, K = r) and
// V = Xhat dH (M = 32 C, N = r, K = p).  One bf16 dH tile [p][r] in the 128-byte-swizzled layout
// is the K-major B operand of the first and the MN-major B operand of the second; the xhat /
// bhat rows and the d_xhat / d_bhat rows of the stage come by TMA.  The epilogue (lanes = rows
// (t, c), four threads per row) adds sc_t U / sc_t V to the gradient rows in shared memory and
// accumulates omega; the copy warp writes the updated rows back with tensor stores.
//
// Warp roles: 0 TMA, 1 MMA, 2-17 epilogue, 18-19 builders.  The builders prepare the next item
// (bf16 dH tile, sc_t, D_n and <dH, h_-(n)>, double-buffered by item parity) while the epilogue
// works on the current one, so the item boundary costs no global-load latency.  Every wait is
// bounded; a timeout sets the workspace error word and the CTA winds down.
#include <cuda.h>

#include "common.cuh"
#include "fast.h"
#include "fast_common.cuh"
#include "prof.h"
#include "tc.cuh"

namespace fastcorr {

using namespace fastk;

constexpr int NEW = 16;                    // epilogue warps: four per TMEM lane quarter
constexpr int NBW = 2;                     // builder warps
constexpr int NTHR = (2 + NEW + NBW) * 32;
static_assert(NBW == 2, "the epilogue sums two dot partials");
constexpr int NS = 2;                      // stages
constexpr uint32_t SLOT = 16384;           // 128 rows x 128 B
// xhat | bhat r 0..63 | bhat r 64..127 | d_xhat | d_bhat r 0..63 | d_bhat r 64..127: the gradient
// rows come in with the stage and go back out by tensor stores once the epilogue updated them
constexpr uint32_t STAGE = 6 * SLOT;
constexpr uint32_t SL_DX = 3, SL_DB = 4;   // slot indices of d_xhat / d_bhat
constexpr uint32_t DHT = 16384;            // dH tile: 64 rows x 2 blocks x 128 B
constexpr uint32_t OFF_DH = NS * STAGE;    // 2 dH tiles
constexpr uint32_t OFF_SC = OFF_DH + 2 * DHT;   // sc_t, 2 items x 64 fp32
constexpr uint32_t OFF_OM = OFF_SC + 512;       // omega of the item, 64 fp32
constexpr uint32_t OFF_OMR = OFF_OM + 256;      // <xhat, U> of the stage rows: [stage parity][128 rows] fp32
constexpr uint32_t OFF_MISC = OFF_OMR + 1024;   // dot partials [item][builder warp], then D_n [item]
constexpr uint32_t OFF_CTL = OFF_MISC + 64;
constexpr uint32_t SMEM_BYTES = OFF_CTL + 128 + 1024;
static_assert(OFF_DH % 1024 == 0 && STAGE % 1024 == 0, "swizzled tiles");
static_assert(SMEM_BYTES <= 232448, "shared memory");

struct Ctl {
    uint64_t full[NS], upd[NS];  // upd: the epilogue has updated the stage's gradient rows
    uint64_t accfull[2], accfree[2];
    uint64_t dhfull[2], dhfree[2];
    uint64_t scfree[2];  // the epilogue has read the item's sc_t, D_n and dot
    uint64_t fin;
    uint32_t tbase;
    int abort;
};
static_assert(sizeof(Ctl) <= 128, "control block");

constexpr uint32_t TM_BUF = 256;  // per accumulator buffer: U at +0 (64 columns), V at +64 (r columns)

struct CItem {
    int bb, hh, n;
    int hd, grp;  // the caller's head and the 64-row group of hh (MMParams::groups)
};

__host__ __device__ inline int count_corr(const MMParams& P) {
    int c = 0;
    for (int bb = 0; bb < P.b; ++bb) {
        const int pr = mm_processed(P, bb);
        c += P.h * (pr > 1 ? pr - 1 : 0);
    }
    return c;
}

// Item -> (batch row, head, chunk) over the chunks followed by another processed chunk.
__device__ inline CItem decode(const MMParams& P, int item) {
    int bb = 0, base = 0;
    for (; bb < P.b - 1; ++bb) {
        const int pr = mm_processed(P, bb);
        const int cnt = P.h * (pr > 1 ? pr - 1 : 0);
        if (item < base + cnt) break;
        base += cnt;
    }
    const int pr = mm_processed(P, bb);
    const int per = pr > 1 ? pr - 1 : 1;
    const int rem = item - base;
    CItem I;
    I.bb = bb;
    I.hh = rem / per;
    I.n = rem - I.hh * per;
    I.hd = I.hh / P.groups;
    I.grp = I.hh - I.hd * P.groups;
    return I;
}

__device__ __forceinline__ int range_begin(int items, int cta) { return (int)(((int64_t)cta * items) / gridDim.x); }

__device__ __forceinline__ void fail(Ctl* ctl, int* err, int code) {
    ctl->abort = 1;
    atomicExch(err, code);
}

struct CorrArgs {
    FastArgs F;        // problem, Hc (carries), err
    const float* da;   // [b,s,h]
    const float* E;    // [b,h,nc,p,r] dH(n+1) per chunk
    __nv_bfloat16* dx;
    __nv_bfloat16* db;
    float* dda;        // with row groups: one [b,s,h] slice per group, summed afterwards
};

__global__ void __launch_bounds__(NTHR, 1)
    tc_corr_kernel(const __grid_constant__ CorrArgs B, const __grid_constant__ CUtensorMap tmx32,
                   const __grid_constant__ CUtensorMap tmb32, const __grid_constant__ CUtensorMap tmdx32,
                   const __grid_constant__ CUtensorMap tmdb32) {
    extern __shared__ unsigned char smraw[];
    unsigned char* sm = smraw + ((1024u - (tc::smem_u32(smraw) & 1023u)) & 1023u);
    Ctl* ctl = reinterpret_cast<Ctl*>(sm + OFF_CTL);
    const FastArgs& A = B.F;
    const MMParams& P = A.P;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int R = P.r, C = P.C;
    const int items = count_corr(P);
    const int it0 = range_begin(items, blockIdx.x), it1 = range_begin(items, blockIdx.x + 1);
    const int TPS = corr_tps(P);                // tokens per stage: rows TPS * C <= 128
    const uint32_t rows = (uint32_t)TPS * C;

    // rows past 32 C of the stage slots, the r >= 64 half (r = 64) and omega start at zero
    for (uint32_t i = tid; i < OFF_CTL / 16; i += NTHR) reinterpret_cast<uint4*>(sm)[i] = make_uint4(0, 0, 0, 0);
    if (tid == 0) {
        for (int s = 0; s < NS; ++s) {
            tc::mbar_init(&ctl->full[s], 1);
            tc::mbar_init(&ctl->upd[s], NEW);
        }
        for (int i = 0; i < 2; ++i) {
            tc::mbar_init(&ctl->accfull[i], 1);
            tc::mbar_init(&ctl->accfree[i], NEW);
            tc::mbar_init(&ctl->dhfull[i], NBW);
            tc::mbar_init(&ctl->dhfree[i], 1);
            tc::mbar_init(&ctl->scfree[i], 1);
        }
        tc::mbar_init(&ctl->fin, 1);
        ctl->abort = 0;
        tc::fence_barrier_init();
    }
    if (warp == 0) {
        tc::tmem_alloc(&ctl->tbase, 512);
        tc::tmem_relinquish();
    }
    tc::fence_proxy_async_smem();
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tbase = ctl->tbase;
    volatile int* abort = &ctl->abort;

    if (warp == 0) {
        // ================================================================ TMA producer
        // Per stage: the xhat / bhat rows and the d_xhat / d_bhat rows of TPS tokens in; before a
        // slot is reused, the stage it held goes back out (the updated gradient rows) by tensor
        // stores, whose reads of the slot complete before the new loads are issued.
        if (lane == 0) {
            uint32_t q = 0;
            bool ok = true;
            // global row and head of the stage each slot holds, and the d_bhat row and head (with
            // row groups d_bhat goes to one [b*s] slice per group: the map's rows are group-major)
            int srow[NS] = {0, 0}, shh[NS] = {0, 0}, sbrow[NS] = {0, 0}, shd[NS] = {0, 0};
            auto store_back = [&](uint32_t qq) -> bool {
                const uint32_t s = qq % NS;
                if (!tc::mbar_wait(&ctl->upd[s], (qq / NS) & 1, abort)) return false;
                unsigned char* stg = sm + s * STAGE;
                tc::tma_store_4d(&tmdx32, 0, shh[s], 0, srow[s], stg + SL_DX * SLOT);
                for (int a = 0; a < (R + 63) / 64; ++a)
                    tc::tma_store_4d(&tmdb32, 64 * a, shd[s], 0, sbrow[s], stg + (SL_DB + a) * SLOT);
                tc::bulk_commit();
                tc::bulk_wait_read0();
                return true;
            };
            for (int it = it0; it < it1 && ok; ++it) {
                const CItem I = decode(P, it);
                for (int st = 0; st < FL / TPS; ++st, ++q) {
                    const uint32_t s = q % NS;
                    if (q >= NS && !(ok = store_back(q - NS))) break;
                    unsigned char* stg = sm + s * STAGE;
                    tc::mbar_arrive_expect_tx(&ctl->full[s], 2u * rows * 128u * (1u + (uint32_t)(R + 63) / 64u));
                    const int row = I.bb * P.s + I.n * FL + st * TPS;
                    const int brow = I.grp * P.b * P.s + row;
                    tc::tma_load_4d(stg, &tmx32, 0, I.hh, 0, row, &ctl->full[s]);
                    tc::tma_load_4d(stg + SL_DX * SLOT, &tmdx32, 0, I.hh, 0, row, &ctl->full[s]);
                    for (int a = 0; a < (R + 63) / 64; ++a) {
                        tc::tma_load_4d(stg + (1 + a) * SLOT, &tmb32, 64 * a, I.hd, 0, row, &ctl->full[s]);
                        tc::tma_load_4d(stg + (SL_DB + a) * SLOT, &tmdb32, 64 * a, I.hd, 0, brow, &ctl->full[s]);
                    }
                    srow[s] = row;
                    shh[s] = I.hh;
                    sbrow[s] = brow;
                    shd[s] = I.hd;
                }
            }
            // the last stages go out too
            for (uint32_t qq = q >= NS ? q - NS : 0; ok && qq < q; ++qq) ok = store_back(qq);
            if (!ok) fail(ctl, A.err, 41);
            tc::bulk_wait0();       // every store has completed
            int never = 0;  // every issued copy lands before the CTA exits
            for (uint32_t s = 0; s < NS && q > s; ++s) {
                const uint32_t last = (q - 1 - s) / NS;
                tc::mbar_wait(&ctl->full[s], last & 1, &never, 1u << 20);
            }
        }
    } else if (warp == 1) {
        // ================================================================ MMA issuer
        if (lane == 0) {
            const uint32_t idU = tc::idesc_bf16(128, 64, 0, 0);  // U: A = bhat rows (K = r), B = dH (K-major)
            const uint32_t idV = tc::idesc_bf16(128, R, 0, 1);   // V: A = xhat rows (K = p), B = dH (MN-major)
            const uint32_t s0 = tc::smem_u32(sm), dh0 = tc::smem_u32(sm + OFF_DH);
            uint32_t q = 0, li = 0;
            bool ok = true;
            for (int it = it0; it < it1 && ok; ++it, ++li) {
                const uint32_t ib = li & 1;
                const uint32_t dh = dh0 + ib * DHT;
                if (!(ok = tc::mbar_wait(&ctl->dhfull[ib], (li >> 1) & 1, abort))) break;
                for (int st = 0; st < FL / TPS; ++st, ++q) {
                    const uint32_t s = q % NS, u = q / NS, ab = q & 1, ua = q >> 1;
                    if (!(ok = tc::mbar_wait(&ctl->full[s], u & 1, abort))) break;
                    if (ua >= 1 && !(ok = tc::mbar_wait(&ctl->accfree[ab], (ua - 1) & 1, abort))) break;
                    tc::tc_fence_after();
                    const uint32_t xs = s0 + s * STAGE, bs = xs + SLOT;
                    const uint32_t tu = tbase + ab * TM_BUF, tv = tu + 64;
                    for (int ks = 0; ks < R / 16; ++ks)
                        tc::mma_bf16(tu, tc::sdesc_sw128(bs + (ks >> 2) * SLOT + 32u * (ks & 3), 16, 1024),
                                     tc::sdesc_sw128(dh + (ks >> 2) * 8192u + 32u * (ks & 3), 16, 1024), idU,
                                     ks > 0);
                    for (int ks = 0; ks < 4; ++ks)
                        tc::mma_bf16(tv, tc::sdesc_sw128(xs + 32u * ks, 16, 1024),
                                     tc::sdesc_sw128(dh + 2048u * ks, 8192, 1024), idV, ks > 0);
                    tc::mma_commit(&ctl->accfull[ab]);
                }
                if (ok) tc::mma_commit(&ctl->dhfree[ib]);
            }
            if (!ok) fail(ctl, A.err, 42);
            tc::mma_commit(&ctl->fin);
            int never = 0;  // in-flight MMAs must finish before the TMEM is released
            tc::mbar_wait(&ctl->fin, 0, &never, 1u << 20);
        }
    } else if (warp < 2 + NEW) {
        // ================================================================ epilogue
        const int ew = warp - 2, etid = tid - 64;
        const int qf = ew >> 2;                     // which quarter of the row's columns
        const int k = ((warp & 3) << 5) + lane;     // TMEM lane = stage row (t, c)
        const uint32_t lane_addr = tbase + ((uint32_t)((warp & 3) * 32) << 16);
        const float* misc = reinterpret_cast<const float*>(sm + OFF_MISC);
        const bool row_ok = (uint32_t)k < rows;
        const int tl = k / C;  // the row's token in the stage (rows are (token, channel))
        uint32_t q = 0, li = 0;
        bool ok = true;
        auto check = [&](bool r) {  // the first failed wait stops the whole CTA at once
            if (!r && ok) {
                ok = false;
                fail(ctl, A.err, 43);
            }
        };
        float* om = reinterpret_cast<float*>(sm + OFF_OM);
        float* omr = reinterpret_cast<float*>(sm + OFF_OMR);
        for (int it = it0; it < it1; ++it, ++li) {
            const CItem I = decode(P, it);
            const uint32_t ib = li & 1;
            const float* sc = reinterpret_cast<const float*>(sm + OFF_SC) + ib * 64;
            check(tc::mbar_wait(&ctl->dhfull[ib], (li >> 1) & 1, abort));  // sc, D_n and the dot are ready
            // ---- the stages of TPS tokens
            for (int st = 0; st < FL / TPS; ++st, ++q) {
                const uint32_t s = q % NS, ab = q & 1;
                const int t = st * TPS + tl;
                // this thread's part of the row: U columns [16 qf, 16 qf + 16), V columns [32 qf, 32 qf + 32)
                const bool has_v = 32 * qf < R;
                check(tc::mbar_wait(&ctl->full[s], (q / NS) & 1, abort));  // the stage's rows are read below
                check(tc::mbar_wait(&ctl->accfull[ab], (q >> 1) & 1, abort));
                tc::tc_fence_after();
                const uint32_t tu = lane_addr + ab * TM_BUF, tv = tu + 64;
                float u[16];
                tc::tmem_ld16(tu + 16 * qf, u);
                tc::tmem_wait_ld();
                unsigned char* const stg = sm + s * STAGE;
                // <xhat row, U row> over all p columns, by the row's first-quarter thread alone
                // (one thread, one fixed order: the sum does not depend on timing)
                if (qf == 0) {
                    float w = 0.f;
                    const unsigned char* xr = stg + k * 128;
#pragma unroll 1
                    for (int q2 = 0; q2 < 4; ++q2) {
                        float uq[16];
                        if (q2 == 0) {
#pragma unroll
                            for (int e = 0; e < 16; ++e) uq[e] = u[e];
                        } else {
                            tc::tmem_ld16(tu + 16 * q2, uq);
                            tc::tmem_wait_ld();
                        }
#pragma unroll
                        for (int jj = 0; jj < 2; ++jj) {
                            const int j = 2 * q2 + jj;
                            const uint4 v = *reinterpret_cast<const uint4*>(xr + ((j ^ (k & 7)) << 4));
                            const uint32_t wd[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                w = fmaf(__uint_as_float(wd[e] << 16), uq[8 * jj + 2 * e], w);
                                w = fmaf(__uint_as_float(wd[e] & 0xFFFF0000u), uq[8 * jj + 2 * e + 1], w);
                            }
                        }
                    }
                    if (row_ok) omr[(st & 1) * 128 + k] = w;
                }
                const float scv = sc[t];
                if (row_ok) {  // d_xhat row += sc U, in the stage's d_xhat slot (same layout as xhat)
                    unsigned char* dr = stg + SL_DX * SLOT + k * 128;
#pragma unroll
                    for (int jj = 0; jj < 2; ++jj) {
                        uint4* pw = reinterpret_cast<uint4*>(dr + (((2 * qf + jj) ^ (k & 7)) << 4));
                        uint4 o = *pw;
                        uint32_t* wd = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float lo = __uint_as_float(wd[e] << 16) + scv * u[8 * jj + 2 * e];
                            const float hi = __uint_as_float(wd[e] & 0xFFFF0000u) + scv * u[8 * jj + 2 * e + 1];
                            wd[e] = tc::pack_bf16x2(lo, hi);
                        }
                        *pw = o;
                    }
                }
                if (has_v) {  // d_bhat row += sc V, columns [32 qf, 32 qf + 32): slot qf / 2, chunks 4 (qf & 1) ..
                    unsigned char* br = stg + (SL_DB + (qf >> 1)) * SLOT + k * 128;
#pragma unroll
                    for (int g = 0; g < 2; ++g) {
                        float v[16];
                        tc::tmem_ld16(tv + 32 * qf + 16 * g, v);
                        tc::tmem_wait_ld();
                        if (row_ok) {
#pragma unroll
                            for (int i = 0; i < 2; ++i) {
                                const int j = 4 * (qf & 1) + 2 * g + i;
                                uint4* pw = reinterpret_cast<uint4*>(br + ((j ^ (k & 7)) << 4));
                                uint4 o = *pw;
                                uint32_t* wd = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
                                for (int e = 0; e < 4; ++e) {
                                    const float lo = __uint_as_float(wd[e] << 16) + scv * v[8 * i + 2 * e];
                                    const float hi =
                                        __uint_as_float(wd[e] & 0xFFFF0000u) + scv * v[8 * i + 2 * e + 1];
                                    wd[e] = tc::pack_bf16x2(lo, hi);
                                }
                                *pw = o;
                            }
                        }
                    }
                }
                tc::fence_proxy_async_smem();  // the updated rows are read by the tensor stores
                tc::tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    tc::mbar_arrive(&ctl->accfree[ab]);
                    tc::mbar_arrive(&ctl->upd[s]);
                }
                // omega of the stage's tokens: each token's C rows, in channel order (the row buffer
                // alternates by stage, so the next stage's rows never overwrite ones still being read)
                named_barrier_sync(1, NEW * 32);
                if (etid < TPS) {
                    const float* pr = omr + (st & 1) * 128 + etid * C;
                    float o = 0.f;
                    for (int c = 0; c < C; ++c) o += pr[c];
                    om[st * TPS + etid] = o;
                }
            }
            named_barrier_sync(1, NEW * 32);  // omega of every token is in
            // ---- d_da_s += D_n <dH, h_-> + sum_{j<s} sc_j omega_j
            if (etid < FL) {
                const float base = misc[2 * NBW + ib] * (misc[NBW * ib] + misc[NBW * ib + 1]);
                float pre = 0.f;
                for (int j = 0; j < etid; ++j) pre = fmaf(sc[j], om[j], pre);
                B.dda[(int64_t)I.grp * P.b * P.s * P.heads + off_da(P, I.bb, I.n * FL + etid, I.hd)] += base + pre;
            }
            named_barrier_sync(1, NEW * 32);  // sc / D_n / omega / dot read: free for the next items
            if (etid == 0) tc::mbar_arrive(&ctl->scfree[ib]);
        }
    } else {
        // ================================================================ builders
        // Item by item, into the buffers of the item's parity once the MMAs (dH tile) and the
        // epilogue (sc_t, D_n, dot) of the item two back are done with them: the bf16 dH tile
        // [p][r] in the 128-byte-swizzled layout, this warp's part of <dH, h_-(n)>, and (warp 0)
        // the decay weights sc_t = exp(a_last - a_t) and D_n = exp(a_last).
        const int bw = warp - 2 - NEW, bt = tid - (2 + NEW) * 32;
        float* misc = reinterpret_cast<float*>(sm + OFF_MISC);
        uint32_t li = 0;
        bool ok = true;
        for (int it = it0; it < it1 && ok; ++it, ++li) {
            const CItem I = decode(P, it);
            const uint32_t ib = li & 1;
            if (li >= 2 && !(ok = tc::mbar_wait(&ctl->dhfree[ib], ((li - 2) >> 1) & 1, abort) &&
                                  tc::mbar_wait(&ctl->scfree[ib], ((li - 2) >> 1) & 1, abort)))
                break;
            if (bw == 0) {  // all 64 tokens of the chunk are valid
                float* sc = reinterpret_cast<float*>(sm + OFF_SC) + ib * 64;
                const int t0 = 2 * lane, t1 = t0 + 1;
                const float v0 = B.da[off_da(P, I.bb, I.n * FL + t0, I.hd)];
                const float v1 = B.da[off_da(P, I.bb, I.n * FL + t1, I.hd)];
                float sum = v0 + v1;
#pragma unroll
                for (int off = 1; off < 32; off <<= 1) {
                    const float o = __shfl_up_sync(0xffffffffu, sum, off);
                    if (lane >= off) sum += o;
                }
                const float alast = __shfl_sync(0xffffffffu, sum, 31);
                sc[t1] = __expf(alast - sum);
                sc[t0] = __expf(alast - (sum - v1));
                if (lane == 0) misc[2 * NBW + ib] = __expf(alast);
            }
            unsigned char* dht = sm + OFF_DH + ib * DHT;
            const float* src = B.E + off_carry(P, I.bb, I.hh, I.n);
            const float* hin = A.Hc + off_carry(P, I.bb, I.hh, I.n);
            float dot = 0.f;
            constexpr int NB = NBW * 32, PER = 64 * 16 / NB, GRP = 4;
            for (int i0 = 0; i0 < PER; i0 += GRP) {
                float4 e[GRP][2], h[GRP][2];
#pragma unroll
                for (int g = 0; g < GRP; ++g) {  // the group's loads are all in flight together
                    const int id = (i0 + g) * NB + bt;
                    const int pp = id >> 4, col = 64 * ((id >> 3) & 1) + 8 * (id & 7);
                    const bool in = col < R;
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        e[g][hh] = in ? *reinterpret_cast<const float4*>(src + pp * R + col + 4 * hh)
                                      : make_float4(0.f, 0.f, 0.f, 0.f);
                        h[g][hh] = in ? *reinterpret_cast<const float4*>(hin + pp * R + col + 4 * hh)
                                      : make_float4(0.f, 0.f, 0.f, 0.f);
                    }
                }
#pragma unroll
                for (int g = 0; g < GRP; ++g) {
                    const int id = (i0 + g) * NB + bt;
                    const int pp = id >> 4, blk = (id >> 3) & 1, j = id & 7;
                    const float4 e0 = e[g][0], e1 = e[g][1], h0 = h[g][0], h1 = h[g][1];
                    dot += e0.x * h0.x + e0.y * h0.y + e0.z * h0.z + e0.w * h0.w;
                    dot += e1.x * h1.x + e1.y * h1.y + e1.z * h1.z + e1.w * h1.w;
                    uint4 w;
                    w.x = tc::pack_bf16x2(e0.x, e0.y);
                    w.y = tc::pack_bf16x2(e0.z, e0.w);
                    w.z = tc::pack_bf16x2(e1.x, e1.y);
                    w.w = tc::pack_bf16x2(e1.z, e1.w);
                    *reinterpret_cast<uint4*>(dht + tc::sw128_chunk(64, blk, pp, j)) = w;
                }
            }
            dot = warp_sum(dot);
            if (lane == 0) misc[NBW * ib + bw] = dot;
            tc::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&ctl->dhfull[ib]);
        }
        if (!ok) fail(ctl, A.err, 44);
    }
    // ---- teardown
    tc::tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc::tc_fence_after();
        tc::tmem_dealloc(tbase, 512);
    }
}

}  // namespace fastcorr

namespace fastk {

cudaError_t launch_tc_corr(const FastArgs& fa, const float* da, const float* E, void* dx, void* db, float* dda,
                           const TensorMaps& maps, cudaStream_t st) {
    using namespace fastcorr;
    const int items = count_corr(fa.P);
    if (items == 0) return cudaSuccess;
    CorrArgs a;
    a.F = fa;
    a.da = da;
    a.E = E;
    a.dx = static_cast<__nv_bfloat16*>(dx);
    a.db = static_cast<__nv_bfloat16*>(db);
    a.dda = dda;
    const int grid = items < sm_count() ? items : sm_count();
    cudaError_t e = mm_allow_smem(reinterpret_cast<const void*>(tc_corr_kernel), (int)SMEM_BYTES);
    if (e != cudaSuccess) return e;
    mm_prof_mark(KID_FAST_CORRECT, 1, st);
    tc_corr_kernel<<<grid, NTHR, SMEM_BYTES, st>>>(a, maps.x32, maps.b32, maps.dx32, maps.db32);
    mm_prof_mark(KID_FAST_CORRECT, 0, st);
    return cudaGetLastError();
}

}  // namespace fastk
