// fast_end.cu -- chunk-end states of the tensor-core path, one GEMM per chunk:
//
//   Delta_n = sum_{t < T_n} sum_c exp(a_last - a_t) xhat_{t,c} (x) bhat_{t,c},   D_n = exp(a_last)
//
// (a_t = inclusive cumulative sum of da inside the chunk).  This is the state a chunk reaches
// from a zero carry, i.e. the per-chunk part of "boundary_carries" in "mamba3/moments/backward.rs";
// written as a contraction over K = (token, channel) it is a single M = r, N = p, K = 64 C
// product instead of 64 dependent token steps.
//
// Operands per 8-token stage, loaded by TMA in the 128-byte-swizzled layout:
//   B operand  xhat rows (t, c) x p  (MN-major, N = p = 64), scaled in place by exp(a_last - a_t)
//              (zero for t >= T_n) by the four epilogue warps before the tensor core reads it;
//   A operand  bhat rows (t, c) x r  (MN-major, M = r: two 64-row blocks; the second stays zero
//              when r = 64).
// The fp32 accumulator D[r][p] lives in tensor memory (two 64-column buffers so that one chunk's
// epilogue overlaps the next chunk's products); the epilogue writes Delta_n[p][r] with lanes = r.
//
// Warp roles: 0 TMA, 1 MMA, 2-5 scaling + epilogue.  Every wait is bounded; a timeout sets the
// workspace error word and the CTA winds down.
#include <cuda.h>

#include "common.cuh"
#include "fast.h"
#include "fast_common.cuh"
#include "prof.h"
#include "tc.cuh"

namespace fastend {

using namespace fastk;

constexpr int NTHR = 192;
constexpr int TPS = 8;                      // tokens per stage
constexpr int NS = 4;                       // stages
constexpr uint32_t SLOT = 8192;             // 64 rows x 128 B
constexpr uint32_t STAGE = 3 * SLOT + 1024; // xhat | bhat half 0 | bhat half 1 | da of the item
constexpr uint32_t OFF_W = NS * STAGE;      // 4 warps x 64 fp32 decay weights
constexpr uint32_t OFF_CTL = OFF_W + 1024;
constexpr uint32_t SMEM_BYTES = OFF_CTL + 256 + 1024;
static_assert(STAGE % 1024 == 0, "swizzled slots");
static_assert(2 * SMEM_BYTES <= 228 * 1024, "two CTAs per SM");

struct Ctl {
    uint64_t full[NS], scaled[NS], empty[NS];
    uint64_t accfull[2], accfree[2];
    uint64_t fin;
    uint64_t never_done;  // nothing arrives on it: the failure-path test waits for it
    uint32_t tbase;
    int abort;
};
static_assert(sizeof(Ctl) <= 256, "control block");

struct EItem {
    int bb, hh, n, T, proc;
    int hd;  // the caller's head (hh is a 64-row group of it, MMParams::groups)
};

__host__ __device__ inline int count_chunks(const MMParams& P) {
    int c = 0;
    for (int bb = 0; bb < P.b; ++bb) c += P.h * mm_processed(P, bb);
    return c;
}

// Item -> (batch row, head, chunk); chunks of one (row, head) are consecutive items.
__device__ inline EItem decode(const MMParams& P, int item) {
    int bb = 0, base = 0;
    for (; bb < P.b - 1; ++bb) {
        const int cnt = P.h * mm_processed(P, bb);
        if (item < base + cnt) break;
        base += cnt;
    }
    EItem I;
    I.bb = bb;
    I.proc = mm_processed(P, bb);
    const int rem = item - base;
    const int pr = I.proc > 0 ? I.proc : 1;
    I.hh = rem / pr;
    I.n = rem - I.hh * pr;
    I.hd = I.hh / P.groups;
    I.T = mm_chunk_rows(P, bb, I.n);
    return I;
}

__device__ __forceinline__ int range_begin(int items, int cta) { return (int)(((int64_t)cta * items) / gridDim.x); }

__device__ __forceinline__ void fail(Ctl* ctl, int* err, int code) {
    ctl->abort = 1;
    atomicExch(err, code);
}

__global__ void __launch_bounds__(NTHR, 2)
    tc_end_kernel(const __grid_constant__ FastArgs A, const __grid_constant__ CUtensorMap tmx8,
                  const __grid_constant__ CUtensorMap tmb8, const __grid_constant__ CUtensorMap tmd64) {
    extern __shared__ unsigned char smraw[];
    unsigned char* sm = smraw + ((1024u - (tc::smem_u32(smraw) & 1023u)) & 1023u);
    Ctl* ctl = reinterpret_cast<Ctl*>(sm + OFF_CTL);
    const MMParams& P = A.P;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int R = P.r, C = P.C;
    const int items = count_chunks(P);
    const int it0 = range_begin(items, blockIdx.x), it1 = range_begin(items, blockIdx.x + 1);
    const uint32_t rows = (uint32_t)TPS * C;             // K rows a stage holds
    const uint32_t ksteps = (rows + 15) / 16;

    // zero the stage slots: rows past TPS*C and the second bhat block (r = 64) must read as zero
    for (uint32_t i = tid; i < NS * STAGE / 16; i += NTHR) reinterpret_cast<uint4*>(sm)[i] = make_uint4(0, 0, 0, 0);
    if (tid == 0) {
        for (int s = 0; s < NS; ++s) {
            tc::mbar_init(&ctl->full[s], 1);
            tc::mbar_init(&ctl->scaled[s], 4);
            tc::mbar_init(&ctl->empty[s], 1);
        }
        for (int i = 0; i < 2; ++i) {
            tc::mbar_init(&ctl->accfull[i], 1);
            tc::mbar_init(&ctl->accfree[i], 4);
        }
        tc::mbar_init(&ctl->fin, 1);
        tc::mbar_init(&ctl->never_done, 1);
        ctl->abort = 0;
        tc::fence_barrier_init();
    }
    if (warp == 0) {
        tc::tmem_alloc(&ctl->tbase, 128);
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
        if (lane == 0) {
            uint32_t q = 0;
            bool ok = true;
            for (int it = it0; it < it1 && ok; ++it) {
                const EItem I = decode(P, it);
                const int nst = (I.T + TPS - 1) / TPS;
                for (int st = 0; st < nst; ++st, ++q) {
                    const uint32_t s = q % NS, u = q / NS;
                    if (u >= 1 && !(ok = tc::mbar_wait(&ctl->empty[s], (u - 1) & 1, abort))) break;
                    unsigned char* stg = sm + s * STAGE;
                    if (st == 0 && !da_by_tma(P)) {
                        // this head's da of the chunk, into the positions the 4-head copy would fill,
                        // before the arrival that publishes the stage
                        float* dst = reinterpret_cast<float*>(stg + 3 * SLOT);
                        const float* src = A.da + ((int64_t)I.bb * P.s + I.n * FL) * P.heads + I.hd;
                        for (int t = 0; t < I.T; ++t) dst[t * 4 + (I.hd & 3)] = src[(int64_t)t * P.heads];
                    }
                    const uint32_t bytes =
                        rows * 128u * (1u + (uint32_t)(R + 63) / 64u) + ((st == 0 && da_by_tma(P)) ? 1024u : 0u);
                    tc::mbar_arrive_expect_tx(&ctl->full[s], bytes);
                    const int row = I.bb * P.s + I.n * FL + st * TPS;
                    tc::tma_load_4d(stg, &tmx8, 0, I.hh, 0, row, &ctl->full[s]);
                    for (int a = 0; a < (R + 63) / 64; ++a)
                        tc::tma_load_4d(stg + (1 + a) * SLOT, &tmb8, 64 * a, I.hd, 0, row, &ctl->full[s]);
                    if (st == 0 && da_by_tma(P))
                        tc::tma_load_2d(stg + 3 * SLOT, &tmd64, I.hd & ~3, I.bb * P.s + I.n * FL, &ctl->full[s]);
                }
            }
            if (!ok) fail(ctl, A.err, 31);
            // every issued copy must land before the CTA exits (own bounded wait)
            int never = 0;
            for (uint32_t s = 0; s < NS && q > s; ++s) {
                const uint32_t last = (q - 1 - s) / NS;
                tc::mbar_wait(&ctl->full[s], last & 1, &never, 1u << 20);
            }
        }
    } else if (warp == 1) {
        // ================================================================ MMA issuer
        if (lane == 0) {
            const uint32_t idesc = tc::idesc_bf16(128, 64, 1, 1);
            const uint32_t s0 = tc::smem_u32(sm);
            uint32_t q = 0, li = 0;
            bool ok = true;
            for (int it = it0; it < it1 && ok; ++it, ++li) {
                const EItem I = decode(P, it);
                const int nst = (I.T + TPS - 1) / TPS;
                const uint32_t ab = li & 1;
                if (li >= 2 && !(ok = tc::mbar_wait(&ctl->accfree[ab], ((li - 2) >> 1) & 1, abort))) break;
                for (int st = 0; st < nst; ++st, ++q) {
                    const uint32_t s = q % NS, u = q / NS;
                    if (!(ok = tc::mbar_wait(&ctl->scaled[s], u & 1, abort))) break;
                    tc::tc_fence_after();
                    const uint32_t xs = s0 + s * STAGE, bs = xs + SLOT;
                    for (uint32_t ks = 0; ks < ksteps; ++ks)
                        tc::mma_bf16(tbase + ab * 64, tc::sdesc_sw128(bs + ks * 2048u, SLOT, 1024),
                                     tc::sdesc_sw128(xs + ks * 2048u, SLOT, 1024), idesc, (st > 0 || ks > 0) ? 1u : 0u);
                    tc::mma_commit(&ctl->empty[s]);
                }
                if (ok) tc::mma_commit(&ctl->accfull[ab]);
            }
            if (!ok) fail(ctl, A.err, 32);
            tc::mma_commit(&ctl->fin);
            int never = 0;  // in-flight MMAs must finish before the TMEM is released
            tc::mbar_wait(&ctl->fin, 0, &never, 1u << 20);
        }
    } else {
        // ================================================================ scaling + epilogue
        const int cw = warp - 2;
        const int m = ((warp & 3) << 5) + lane;  // TMEM lane = r
        const uint32_t lane_addr = tbase + ((uint32_t)((warp & 3) * 32) << 16);
        float* wsm = reinterpret_cast<float*>(sm + OFF_W) + cw * 64;
        uint32_t q = 0, li = 0;
        bool ok = true;
        auto check = [&](bool r) {  // the first failed wait stops the whole CTA at once
            if (!r && ok) {
                ok = false;
                fail(ctl, A.err, 33);
            }
        };
        // failure-path test: a wait that gives up after a few thousand polls, then the CTA winds
        // down like after any other timeout
        if (A.test_wait_timeout) check(tc::mbar_wait(&ctl->never_done, 0, abort, 1u << 12));
        for (int it = it0; it < it1; ++it, ++li) {
            const EItem I = decode(P, it);
            const int nst = (I.T + TPS - 1) / TPS;
            const uint32_t ab = li & 1;
            for (int st = 0; st < nst; ++st, ++q) {
                const uint32_t s = q % NS, u = q / NS;
                check(tc::mbar_wait(&ctl->full[s], u & 1, abort));
                unsigned char* stg = sm + s * STAGE;
                if (st == 0) {
                    // decay weights of the chunk: inclusive cumulative sum of da by a warp scan
                    const float* da = reinterpret_cast<const float*>(stg + 3 * SLOT);
                    const int t0 = 2 * lane, t1 = t0 + 1;
                    const float v0 = t0 < I.T ? da[t0 * 4 + (I.hd & 3)] : 0.f;
                    const float v1 = t1 < I.T ? da[t1 * 4 + (I.hd & 3)] : 0.f;
                    float sum = v0 + v1;
#pragma unroll
                    for (int off = 1; off < 32; off <<= 1) {
                        const float o = __shfl_up_sync(0xffffffffu, sum, off);
                        if (lane >= off) sum += o;
                    }
                    const float a1 = sum, a0 = sum - v1;
                    const float alast = __shfl_sync(0xffffffffu, sum, 31);  // da of t >= T counted as 0
                    wsm[t0] = t0 < I.T ? __expf(alast - a0) : 0.f;
                    wsm[t1] = t1 < I.T ? __expf(alast - a1) : 0.f;
                    if (cw == 0 && lane == 0) A.Dn[((int64_t)I.bb * P.h + I.hh) * P.nc + I.n] = __expf(alast);
                    __syncwarp();
                }
                // scale the xhat rows of the stage in place (rows are (token, channel))
                const uint32_t units = rows * 8u;
                for (uint32_t un = (uint32_t)(cw * 32 + lane); un < units; un += 128u) {
                    const uint32_t row = un >> 3;
                    const float w = wsm[st * TPS + (int)(row / (uint32_t)C)];
                    uint4* p = reinterpret_cast<uint4*>(stg + un * 16u);
                    uint4 v = *p;
                    uint32_t* wd = reinterpret_cast<uint32_t*>(&v);
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const float lo = __uint_as_float(wd[j] << 16), hi = __uint_as_float(wd[j] & 0xFFFF0000u);
                        wd[j] = tc::pack_bf16x2(w * lo, w * hi);
                    }
                    *p = v;
                }
                tc::fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) tc::mbar_arrive(&ctl->scaled[s]);
            }
            // epilogue: D[r][p] -> Delta_n[p][r] (the last processed chunk's end state is never read)
            check(tc::mbar_wait(&ctl->accfull[ab], (li >> 1) & 1, abort));
            tc::tc_fence_after();
            const bool store = I.n + 1 < I.proc && m < R;
            float* dst = A.Hc + off_carry(P, I.bb, I.hh, I.n) + m;
#pragma unroll
            for (int g = 0; g < 4; ++g) {
                float v[16];
                tc::tmem_ld16(lane_addr + ab * 64 + 16 * g, v);
                tc::tmem_wait_ld();
                if (store) {
#pragma unroll
                    for (int e = 0; e < 16; ++e) dst[(int64_t)(16 * g + e) * R] = v[e];
                }
            }
            tc::tc_fence_before();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&ctl->accfree[ab]);
        }
    }
    // ---- teardown
    tc::tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc::tc_fence_after();
        tc::tmem_dealloc(tbase, 128);
    }
}

}  // namespace fastend

namespace fastk {

cudaError_t launch_tc_end(const FastArgs& fa, const TensorMaps& maps, cudaStream_t st) {
    using namespace fastend;
    const int items = count_chunks(fa.P);
    if (items == 0) return cudaSuccess;
    const int grid = items < 2 * sm_count() ? items : 2 * sm_count();
    cudaError_t e = mm_allow_smem(reinterpret_cast<const void*>(tc_end_kernel), (int)SMEM_BYTES);
    if (e != cudaSuccess) return e;
    mm_prof_mark(KID_FAST_END, 1, st);
    tc_end_kernel<<<grid, NTHR, SMEM_BYTES, st>>>(fa, maps.x8, maps.b8, maps.da64);
    mm_prof_mark(KID_FAST_END, 0, st);
    return cudaGetLastError();
}

}  // namespace fastk
