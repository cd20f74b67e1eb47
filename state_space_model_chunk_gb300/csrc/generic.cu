// generic.cu -- SIMT fp32 kernels of the state-moments operator, for every shape.
//
// Chunk-parallel decomposition (burn-mamba "mamba3/moments/backward.rs" module header and
// boundary_carries; "mamba3/moments/recalculated.rs" moments_phys_fwd):
//   forward : chunk_end  -> carry_scan -> fwd_chunk (m2/m1)
//   backward: chunk_end  -> carry_scan -> bwd_chunk (local VJPs, carry cotangent e_n)
//             -> cot_scan (dH(n) = e_n + D_n dH(n+1)) -> correct (adds the dH terms)
// Inside a chunk the states follow the token recurrence h_t = e^{da_t} h_{t-1} + W_t, which is
// the chunk form h~[t] = d_t h_- + sum_{j<=t} L[t,j] W_j unrolled; nothing of the state
// trajectory outlives one chunk (the backward keeps one chunk in a per-block scratch slot).
#include "common.cuh"
#include "generic.h"
#include "prof.h"

namespace {

constexpr int NT = 256;      // threads per block of every SIMT kernel
constexpr int EPT = 64;      // max state elements per thread (p * r <= 16384)

// Per-token rotation parameters staged in shared memory: cos/sin of the angles (complex)
// or the quaternions.
__device__ void stage_rot(const MMParams& P, const float* rot, int bb, int t, int hh, float* cs,
                          float* sn, float* q) {
    if (P.rw == 0 || rot == nullptr) return;
    const float* src = rot + off_rot(P, bb, t, hh);
    if (P.rot == ROT_QUAT) {
        for (int i = threadIdx.x; i < 4 * P.J; i += blockDim.x) q[i] = src[i];
    } else {
        for (int i = threadIdx.x; i < P.na; i += blockDim.x) {
            float s_, c_;
            sincosf(src[i], &s_, &c_);
            cs[i] = c_;
            sn[i] = s_;
        }
    }
}

__device__ __forceinline__ float qcomp(const float* Q, const float* v, int comp, bool conjq) {
    float qw = Q[0], qx = conjq ? -Q[1] : Q[1], qy = conjq ? -Q[2] : Q[2], qz = conjq ? -Q[3] : Q[3];
    switch (comp) {
        case 0: return qw * v[0] - qx * v[1] - qy * v[2] - qz * v[3];
        case 1: return qw * v[1] + qx * v[0] + qy * v[3] - qz * v[2];
        case 2: return qw * v[2] - qx * v[3] + qy * v[0] + qz * v[1];
        default: return qw * v[3] + qx * v[2] - qy * v[1] + qz * v[0];
    }
}

// Element k of the rotated row v: de-rotation R(-theta) / Q (x) . when tr == false, its
// transpose R(+theta) / conj(Q) (x) . when tr == true ("rotate_chunk").
__device__ __forceinline__ float rot_elem(const MMParams& P, const float* v, int k, const float* cs,
                                          const float* sn, const float* q, bool tr) {
    if (P.rot == ROT_PAIRWISE) {
        if (k < 2 * P.na) {
            int i = k >> 1;
            float c = cs[i], s = tr ? -sn[i] : sn[i];
            return (k & 1) ? (-s * v[k - 1] + c * v[k]) : (c * v[k] + s * v[k + 1]);
        }
    } else if (P.rot == ROT_HALF) {
        int half = P.r >> 1;
        if (k < P.na) {
            float c = cs[k], s = tr ? -sn[k] : sn[k];
            return c * v[k] + s * v[k + half];
        }
        if (k >= half && k < half + P.na) {
            int i = k - half;
            float c = cs[i], s = tr ? -sn[i] : sn[i];
            return -s * v[i] + c * v[k];
        }
    } else if (P.rot == ROT_QUAT) {
        if (k < 4 * P.J) {
            int blk = k >> 2;
            return qcomp(q + 4 * blk, v + 4 * blk, k & 3, tr);
        }
    }
    return v[k];
}

template <typename T>
__device__ void stage_token(const MMParams& P, const T* xhat, const T* bhat, int bb, int t, int hh,
                            float* xs, float* bs, float xscale) {
    for (int i = threadIdx.x; i < P.C * P.p; i += blockDim.x) {
        int c = i / P.p, pp = i - c * P.p;
        xs[i] = xscale * ld_val(xhat + off_x(P, bb, t, c, hh) + pp);
    }
    for (int i = threadIdx.x; i < P.C * P.r; i += blockDim.x) {
        int c = i / P.r, rr = i - c * P.r;
        bs[i] = ld_val(bhat + off_b(P, bb, t, c, hh) + rr);
    }
}

// ---------------------------------------------------------------- Dsym = d_m2 + d_m2^T
__global__ void k_dsym(const float* __restrict__ dm2, float* __restrict__ dsym, int64_t nbh, int r) {
    int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
    int64_t rr = (int64_t)r * r;
    if (i >= nbh * rr) return;
    int64_t base = (i / rr) * rr;
    int rem = (int)(i - base), a = rem / r, c = rem - a * r;
    dsym[i] = dm2[i] + dm2[base + (int64_t)c * r + a];
}

// ------------------------------------------------------- chunk-end contributions (K1)
// Delta_n = sum_{j,c} exp(a_last - a_j) xhat_jc (x) bhat_jc ; D_n = exp(a_last)
// ("backward.rs", boundary_carries: decay-to-chunk-end contraction).
template <typename T>
__global__ void __launch_bounds__(NT) k_chunk_end(MMParams P, const T* __restrict__ xhat,
                                                  const T* __restrict__ bhat, const float* __restrict__ da,
                                                  float* __restrict__ Hc, float* __restrict__ Dn) {
    const int n = blockIdx.x, hh = blockIdx.y, bb = blockIdx.z;
    const int proc = mm_processed(P, bb);
    if (n >= proc) return;
    extern __shared__ float sm[];
    float* a = sm;
    float* xs = a + P.l;
    float* bs = xs + P.C * P.p;
    if (threadIdx.x == 0) {
        float acc = 0.f;
        for (int j = 0; j < P.l; ++j) {
            acc += da[off_da(P, bb, n * P.l + j, hh)];
            a[j] = acc;
        }
        Dn[((int64_t)bb * P.h + hh) * P.nc + n] = expf(acc);
    }
    __syncthreads();
    if (n == proc - 1) return;  // the last processed chunk's end state is never consumed
    const int pr = P.p * P.r;
    const float alast = a[P.l - 1];
    float acc[EPT];
#pragma unroll
    for (int k = 0; k < EPT; ++k) acc[k] = 0.f;
    for (int j = 0; j < P.l; ++j) {
        stage_token(P, xhat, bhat, bb, n * P.l + j, hh, xs, bs, expf(alast - a[j]));
        __syncthreads();
#pragma unroll
        for (int k = 0; k < EPT; ++k) {
            int e = threadIdx.x + k * NT;
            if (e < pr) {
                int pp = e / P.r, rr = e - pp * P.r;
                float s = 0.f;
                for (int c = 0; c < P.C; ++c) s += xs[c * P.p + pp] * bs[c * P.r + rr];
                acc[k] += s;
            }
        }
        __syncthreads();
    }
    float* out = Hc + off_carry(P, bb, hh, n);
#pragma unroll
    for (int k = 0; k < EPT; ++k) {
        int e = threadIdx.x + k * NT;
        if (e < pr) out[e] = acc[k];
    }
}

// -------------------------------------------------------------- carry scan (K2)
// In place: slot n holds Delta_n on entry and the carry h_-(n) on exit.
// h_-(0) = initial, h_-(n+1) = D_n h_-(n) + Delta_n ("boundary_carries", serial part).
// Each thread owns V consecutive elements of the p x r state (V = 4: float4 when p r % 4 == 0)
// and reads the slots of SCAN_B chunks ahead before the dependent updates, so that a thread keeps
// SCAN_B independent loads in flight.
constexpr int SCAN_T = 128, SCAN_B = 16;

template <int V>
struct Vec;
template <>
struct Vec<1> {
    using T = float;
    __device__ static T zero() { return 0.f; }
    __device__ static T fma(float a, T x, T y) { return fmaf(a, x, y); }
    __device__ static T add(T x, T y) { return x + y; }
};
template <>
struct Vec<4> {
    using T = float4;
    __device__ static T zero() { return make_float4(0.f, 0.f, 0.f, 0.f); }
    __device__ static T fma(float a, T x, T y) {
        return make_float4(fmaf(a, x.x, y.x), fmaf(a, x.y, y.y), fmaf(a, x.z, y.z), fmaf(a, x.w, y.w));
    }
    __device__ static T add(T x, T y) { return make_float4(x.x + y.x, x.y + y.y, x.z + y.z, x.w + y.w); }
};

// The two scans below run down each (b,h)'s chunk slots in batches of SCAN_B, software-pipelined:
// the next batch's loads are issued before the current batch's stores, so that a thread always
// has SCAN_B loads in flight (the loaded and the stored slots of one step never overlap).
template <int V>
__global__ void __launch_bounds__(SCAN_T) k_carry_scan(MMParams P, const float* __restrict__ initial,
                                                       float* __restrict__ Hc, const float* __restrict__ Dn) {
    using VT = typename Vec<V>::T;
    const int hh = blockIdx.y, bb = blockIdx.z;
    const int64_t nv = (int64_t)P.p * P.r / V;
    const int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (e >= nv) return;
    const int proc = mm_processed(P, bb);
    VT H = reinterpret_cast<const VT*>(initial + ((int64_t)bb * P.h + hh) * nv * V)[e];
    const float* D = Dn + ((int64_t)bb * P.h + hh) * P.nc;
    VT* slot0 = reinterpret_cast<VT*>(Hc + off_carry(P, bb, hh, 0)) + e;
    // slot n holds Delta_n on entry and the carry H_n entering chunk n on exit (the last
    // processed chunk's Delta is not needed)
    VT d[SCAN_B], dn[SCAN_B];
#pragma unroll
    for (int j = 0; j < SCAN_B; ++j) d[j] = (j + 1 < proc) ? slot0[(int64_t)j * nv] : Vec<V>::zero();
    for (int n0 = 0; n0 < proc; n0 += SCAN_B) {
#pragma unroll
        for (int j = 0; j < SCAN_B; ++j)
            dn[j] = (n0 + SCAN_B + j + 1 < proc) ? slot0[(int64_t)(n0 + SCAN_B + j) * nv] : Vec<V>::zero();
#pragma unroll
        for (int j = 0; j < SCAN_B; ++j) {
            if (n0 + j < proc) {
                slot0[(int64_t)(n0 + j) * nv] = H;
                H = Vec<V>::fma(D[n0 + j], H, d[j]);
            }
        }
#pragma unroll
        for (int j = 0; j < SCAN_B; ++j) d[j] = dn[j];
    }
}

// ----------------------------------------------------------- forward chunk (K3)
// States by the token recurrence from the chunk's carry, de-rotation, masked moment sums.
// m2 / m1 are accumulated with atomics (zeroed by the host beforehand).
template <typename T>
__global__ void __launch_bounds__(NT) k_fwd_chunk(MMParams P, const T* __restrict__ xhat,
                                                  const T* __restrict__ bhat, const float* __restrict__ da,
                                                  const float* __restrict__ rot, const float* __restrict__ Hc,
                                                  float* __restrict__ m2, float* __restrict__ m1) {
    const int n = blockIdx.x, hh = blockIdx.y, bb = blockIdx.z;
    if (n >= mm_processed(P, bb)) return;
    const int T_ = mm_chunk_rows(P, bb, n);
    const int pr = P.p * P.r;
    extern __shared__ float sm[];
    float* S = sm;
    float* Cb = S + pr;
    float* xs = Cb + pr;
    float* bs = xs + P.C * P.p;
    float* cs = bs + P.C * P.r;
    float* sn = cs + (P.r > 4 ? P.r : 4);
    float* q = sn + (P.r > 4 ? P.r : 4);
    const float* carry = Hc + off_carry(P, bb, hh, n);
    for (int e = threadIdx.x; e < pr; e += NT) S[e] = carry[e];
    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
    const int R16 = (P.r + 15) >> 4;
    float acc[8][8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;
    float m1acc = 0.f;
    for (int t = 0; t < T_; ++t) {
        const int tok = n * P.l + t;
        stage_token(P, xhat, bhat, bb, tok, hh, xs, bs, 1.f);
        stage_rot(P, rot, bb, tok, hh, cs, sn, q);
        const float et = expf(da[off_da(P, bb, tok, hh)]);
        __syncthreads();
        for (int e = threadIdx.x; e < pr; e += NT) {
            int pp = e / P.r, rr = e - pp * P.r;
            float w = 0.f;
            for (int c = 0; c < P.C; ++c) w += xs[c * P.p + pp] * bs[c * P.r + rr];
            S[e] = et * S[e] + w;
        }
        __syncthreads();
        for (int e = threadIdx.x; e < pr; e += NT) {
            int pp = e / P.r, rr = e - pp * P.r;
            Cb[e] = rot_elem(P, S + pp * P.r, rr, cs, sn, q, false);
        }
        __syncthreads();
        for (int pp = 0; pp < P.p; ++pp) {
            const float* row = Cb + pp * P.r;
            float rv[8], cv[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                int ri = ty + 16 * i, ci = tx + 16 * i;
                rv[i] = (i < R16 && ri < P.r) ? row[ri] : 0.f;
                cv[i] = (i < R16 && ci < P.r) ? row[ci] : 0.f;
            }
#pragma unroll
            for (int i = 0; i < 8; ++i)
#pragma unroll
                for (int j = 0; j < 8; ++j) acc[i][j] += rv[i] * cv[j];
            if ((int)threadIdx.x < P.r) m1acc += row[threadIdx.x];
        }
        __syncthreads();
    }
    float* M2 = m2 + ((int64_t)bb * P.h + hh) * P.r * P.r;
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            int ri = ty + 16 * i, ci = tx + 16 * j;
            if (i < R16 && j < R16 && ri < P.r && ci < P.r) atomicAdd(M2 + ri * P.r + ci, acc[i][j]);
        }
    if ((int)threadIdx.x < P.r) atomicAdd(m1 + ((int64_t)bb * P.h + hh) * P.r + threadIdx.x, m1acc);
}

// -------------------------------------------------------- backward chunk, local (K5)
// For one chunk with zero incoming cotangent: recompute the states from the carry into a
// per-block scratch slot, then walk the tokens in reverse with the running cotangent g:
//   d_c = c (D + D^T) + d_m1 ; d_rot ; g += R^T d_c ; d_xhat = g bhat ; d_bhat = g^T xhat ;
//   d_da_t = e_t <g, h_{t-1}> ; g *= e_t.   After the chunk, e_n = g (cotangent of h_-).
template <typename T>
__global__ void __launch_bounds__(NT) k_bwd_chunk(MMParams P, const T* __restrict__ xhat,
                                                  const T* __restrict__ bhat, const float* __restrict__ da,
                                                  const float* __restrict__ rot, const float* __restrict__ Hc,
                                                  const float* __restrict__ dsym, const float* __restrict__ dm1,
                                                  T* __restrict__ dxhat, T* __restrict__ dbhat,
                                                  float* __restrict__ dda, float* __restrict__ drot,
                                                  float* __restrict__ E, float* __restrict__ traj) {
    const int pr = P.p * P.r;
    extern __shared__ float sm[];
    float* Sb = sm;
    float* Cb = Sb + pr;
    float* Db = Cb + pr;
    float* g = Db + pr;
    float* xs = g + pr;
    float* bs = xs + P.C * P.p;
    float* cs = bs + P.C * P.r;
    float* sn = cs + (P.r > 4 ? P.r : 4);
    float* q = sn + (P.r > 4 ? P.r : 4);
    float* red = q + (P.r > 4 ? P.r : 4);
    float* mytraj = traj + (int64_t)blockIdx.x * P.l * pr;
    const int64_t total = (int64_t)P.b * P.h * P.nc;
    for (int64_t job = blockIdx.x; job < total; job += gridDim.x) {
        const int n = (int)(job % P.nc);
        const int hh = (int)((job / P.nc) % P.h);
        const int bb = (int)(job / ((int64_t)P.nc * P.h));
        if (n >= mm_processed(P, bb)) continue;
        const int T_ = mm_chunk_rows(P, bb, n);
        const float* carry = Hc + off_carry(P, bb, hh, n);
        const float* Dsym = dsym + ((int64_t)bb * P.h + hh) * P.r * P.r;
        const float* dM1 = dm1 + ((int64_t)bb * P.h + hh) * P.r;
        // forward recurrence over the chunk, states kept in this block's scratch slot
        for (int e = threadIdx.x; e < pr; e += NT) Sb[e] = carry[e];
        for (int t = 0; t < T_; ++t) {
            const int tok = n * P.l + t;
            stage_token(P, xhat, bhat, bb, tok, hh, xs, bs, 1.f);
            const float et = expf(da[off_da(P, bb, tok, hh)]);
            __syncthreads();
            for (int e = threadIdx.x; e < pr; e += NT) {
                int pp = e / P.r, rr = e - pp * P.r;
                float w = 0.f;
                for (int c = 0; c < P.C; ++c) w += xs[c * P.p + pp] * bs[c * P.r + rr];
                float v = et * Sb[e] + w;
                Sb[e] = v;
                mytraj[(int64_t)t * pr + e] = v;
            }
            __syncthreads();
        }
        for (int e = threadIdx.x; e < pr; e += NT) g[e] = 0.f;
        for (int t = T_ - 1; t >= 0; --t) {
            const int tok = n * P.l + t;
            stage_token(P, xhat, bhat, bb, tok, hh, xs, bs, 1.f);
            stage_rot(P, rot, bb, tok, hh, cs, sn, q);
            const float et = expf(da[off_da(P, bb, tok, hh)]);
            for (int e = threadIdx.x; e < pr; e += NT) Sb[e] = mytraj[(int64_t)t * pr + e];
            __syncthreads();
            for (int e = threadIdx.x; e < pr; e += NT) {
                int pp = e / P.r, rr = e - pp * P.r;
                Cb[e] = rot_elem(P, Sb + pp * P.r, rr, cs, sn, q, false);
            }
            __syncthreads();
            // moments VJP: d_c[p, r2] = d_m1[r2] + sum_r1 c[p, r1] Dsym[r1, r2]
            for (int e = threadIdx.x; e < pr; e += NT) {
                int pp = e / P.r, r2 = e - pp * P.r;
                const float* crow = Cb + pp * P.r;
                float s = dM1[r2];
                for (int r1 = 0; r1 < P.r; ++r1) s += crow[r1] * Dsym[(int64_t)r1 * P.r + r2];
                Db[e] = s;
            }
            __syncthreads();
            // rotation-parameter VJP (sum over the p rows)
            if (P.rw) {
                float* dr = drot + off_rot(P, bb, tok, hh);
                if (P.rot == ROT_QUAT) {
                    for (int i = threadIdx.x; i < 4 * P.J; i += NT) {
                        int blk = i >> 2, comp = i & 3;
                        float s = 0.f;
                        for (int pp = 0; pp < P.p; ++pp) {
                            const float* dcb = Db + pp * P.r + 4 * blk;
                            const float* hb = Sb + pp * P.r + 4 * blk;
                            // (d_c (x) conj(h))[comp], the bilinear-product VJP
                            float hw = hb[0], hx = -hb[1], hy = -hb[2], hz = -hb[3];
                            float aw = dcb[0], ax = dcb[1], ay = dcb[2], az = dcb[3];
                            float v;
                            if (comp == 0) v = aw * hw - ax * hx - ay * hy - az * hz;
                            else if (comp == 1) v = aw * hx + ax * hw + ay * hz - az * hy;
                            else if (comp == 2) v = aw * hy - ax * hz + ay * hw + az * hx;
                            else v = aw * hz + ax * hy - ay * hx + az * hw;
                            s += v;
                        }
                        dr[i] = s;
                    }
                } else {
                    for (int i = threadIdx.x; i < P.na; i += NT) {
                        int ix = (P.rot == ROT_PAIRWISE) ? 2 * i : i;
                        int iy = (P.rot == ROT_PAIRWISE) ? 2 * i + 1 : i + (P.r >> 1);
                        float s = 0.f;
                        for (int pp = 0; pp < P.p; ++pp) {
                            const float* dc = Db + pp * P.r;
                            const float* cc = Cb + pp * P.r;
                            s += dc[ix] * cc[iy] - dc[iy] * cc[ix];
                        }
                        dr[i] = s;
                    }
                }
            }
            // cotangent back to the cache frame
            for (int e = threadIdx.x; e < pr; e += NT) {
                int pp = e / P.r, rr = e - pp * P.r;
                g[e] += rot_elem(P, Db + pp * P.r, rr, cs, sn, q, true);
            }
            __syncthreads();
            for (int i = threadIdx.x; i < P.C * P.p; i += NT) {
                int c = i / P.p, pp = i - c * P.p;
                const float* grow = g + pp * P.r;
                const float* brow = bs + c * P.r;
                float s = 0.f;
                for (int rr = 0; rr < P.r; ++rr) s += grow[rr] * brow[rr];
                st_val(dxhat + off_x(P, bb, tok, c, hh) + pp, s);
            }
            for (int i = threadIdx.x; i < P.C * P.r; i += NT) {
                int c = i / P.r, rr = i - c * P.r;
                const float* xrow = xs + c * P.p;
                float s = 0.f;
                for (int pp = 0; pp < P.p; ++pp) s += g[pp * P.r + rr] * xrow[pp];
                st_val(dbhat + off_b(P, bb, tok, c, hh) + rr, s);
            }
            const float* hprev = (t > 0) ? (mytraj + (int64_t)(t - 1) * pr) : carry;
            float part = 0.f;
            for (int e = threadIdx.x; e < pr; e += NT) part += g[e] * hprev[e];
            float dot = block_sum(part, red);
            if (threadIdx.x == 0) dda[off_da(P, bb, tok, hh)] = et * dot;
            for (int e = threadIdx.x; e < pr; e += NT) g[e] *= et;
            __syncthreads();
        }
        float* En = E + off_carry(P, bb, hh, n);
        for (int e = threadIdx.x; e < pr; e += NT) En[e] = g[e];
        __syncthreads();
    }
}

// ------------------------------------------------ carry-cotangent scan (K6)
// In place: slot n holds e_n on entry and dH(n+1), the cotangent of chunk n's end state, on
// exit.  dH(P) = 0, dH(n) = e_n + D_n dH(n+1), d_initial = dH(0).
template <int V>
__global__ void __launch_bounds__(SCAN_T) k_cot_scan(MMParams P, float* __restrict__ E, const float* __restrict__ Dn,
                                                     float* __restrict__ dinit) {
    using VT = typename Vec<V>::T;
    const int hh = blockIdx.y, bb = blockIdx.z;
    const int64_t nv = (int64_t)P.p * P.r / V;
    const int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (e >= nv) return;
    const int proc = mm_processed(P, bb);
    const float* D = Dn + ((int64_t)bb * P.h + hh) * P.nc;
    VT* slot0 = reinterpret_cast<VT*>(E + off_carry(P, bb, hh, 0)) + e;
    VT dH = Vec<V>::zero();
    VT en[SCAN_B], enn[SCAN_B];
#pragma unroll
    for (int j = 0; j < SCAN_B; ++j) en[j] = (proc - 1 - j >= 0) ? slot0[(int64_t)(proc - 1 - j) * nv] : Vec<V>::zero();
    for (int n0 = proc - 1; n0 >= 0; n0 -= SCAN_B) {
#pragma unroll
        for (int j = 0; j < SCAN_B; ++j)
            enn[j] = (n0 - SCAN_B - j >= 0) ? slot0[(int64_t)(n0 - SCAN_B - j) * nv] : Vec<V>::zero();
#pragma unroll
        for (int j = 0; j < SCAN_B; ++j) {
            if (n0 - j >= 0) {
                slot0[(int64_t)(n0 - j) * nv] = dH;
                dH = Vec<V>::fma(D[n0 - j], dH, en[j]);
            }
        }
#pragma unroll
        for (int j = 0; j < SCAN_B; ++j) en[j] = enn[j];
    }
    reinterpret_cast<VT*>(dinit + ((int64_t)bb * P.h + hh) * nv * V)[e] = dH;
}

// ---------------------------------------------- boundary-cotangent correction (K7)
// Adds the terms of dH = dH(n+1) to chunk n (all of whose tokens are valid):
//   d_xhat_jc += sc_j dH bhat_jc ; d_bhat_jc += sc_j dH^T xhat_jc ;
//   d_da_s    += D_n <dH, h_-> + sum_{j<s} sc_j <dH, W_j>,   sc_j = exp(a_last - a_j).
template <typename T>
__global__ void __launch_bounds__(NT) k_correct(MMParams P, const T* __restrict__ xhat,
                                                const T* __restrict__ bhat, const float* __restrict__ da,
                                                const float* __restrict__ Hc, const float* __restrict__ E,
                                                T* __restrict__ dxhat, T* __restrict__ dbhat,
                                                float* __restrict__ dda) {
    const int n = blockIdx.x, hh = blockIdx.y, bb = blockIdx.z;
    if (n + 1 >= mm_processed(P, bb)) return;
    const int pr = P.p * P.r;
    extern __shared__ float sm[];
    float* dH = sm;
    float* xs = dH + pr;
    float* bs = xs + P.C * P.p;
    float* U = bs + P.C * P.r;
    float* a = U + P.C * P.p;
    float* om = a + P.l;
    float* red = om + P.l;
    const float* src = E + off_carry(P, bb, hh, n);
    const float* hin = Hc + off_carry(P, bb, hh, n);
    float part = 0.f;
    for (int e = threadIdx.x; e < pr; e += NT) {
        float v = src[e];
        dH[e] = v;
        part += v * hin[e];
    }
    if (threadIdx.x == 0) {
        float acc = 0.f;
        for (int j = 0; j < P.l; ++j) {
            acc += da[off_da(P, bb, n * P.l + j, hh)];
            a[j] = acc;
        }
    }
    const float hdot = block_sum(part, red);  // includes a __syncthreads
    const float alast = a[P.l - 1];
    for (int j = 0; j < P.l; ++j) {
        const int tok = n * P.l + j;
        stage_token(P, xhat, bhat, bb, tok, hh, xs, bs, 1.f);
        __syncthreads();
        const float sc = expf(alast - a[j]);
        float om_part = 0.f;
        for (int i = threadIdx.x; i < P.C * P.p; i += NT) {
            int c = i / P.p, pp = i - c * P.p;
            const float* drow = dH + pp * P.r;
            const float* brow = bs + c * P.r;
            float s = 0.f;
            for (int rr = 0; rr < P.r; ++rr) s += drow[rr] * brow[rr];
            U[i] = s;
            om_part += s * xs[i];
            T* dst = dxhat + off_x(P, bb, tok, c, hh) + pp;
            st_val(dst, ld_val(dst) + sc * s);
        }
        for (int i = threadIdx.x; i < P.C * P.r; i += NT) {
            int c = i / P.r, rr = i - c * P.r;
            const float* xrow = xs + c * P.p;
            float s = 0.f;
            for (int pp = 0; pp < P.p; ++pp) s += dH[pp * P.r + rr] * xrow[pp];
            T* dst = dbhat + off_b(P, bb, tok, c, hh) + rr;
            st_val(dst, ld_val(dst) + sc * s);
        }
        float w = block_sum(om_part, red);
        if (threadIdx.x == 0) om[j] = sc * w;
        __syncthreads();
    }
    if (threadIdx.x == 0) {
        const float base = expf(alast) * hdot;
        float pre = 0.f;
        for (int j = 0; j < P.l; ++j) {
            dda[off_da(P, bb, n * P.l + j, hh)] += base + pre;
            pre += om[j];
        }
    }
}

inline int rot_pad(const MMParams& P) { return P.r > 4 ? P.r : 4; }

}  // namespace

// ------------------------------------------------------------------- host launchers
size_t generic_fwd_smem(const MMParams& P) {
    return sizeof(float) * (2 * (size_t)P.p * P.r + P.C * (P.p + P.r) + 3 * rot_pad(P));
}
size_t generic_bwd_smem(const MMParams& P) {
    return sizeof(float) * (4 * (size_t)P.p * P.r + P.C * (P.p + P.r) + 3 * rot_pad(P) + 32);
}
size_t generic_correct_smem(const MMParams& P) {
    return sizeof(float) * ((size_t)P.p * P.r + P.C * (2 * P.p + P.r) + 2 * P.l + 32);
}
size_t generic_end_smem(const MMParams& P) { return sizeof(float) * (P.l + P.C * (P.p + P.r)); }

bool generic_supported(const MMParams& P, int smem_limit) {
    if ((int64_t)P.p * P.r > NT * EPT || P.r > 128) return false;
    if ((int)generic_bwd_smem(P) > smem_limit || (int)generic_fwd_smem(P) > smem_limit) return false;
    if ((int)generic_correct_smem(P) > smem_limit || (int)generic_end_smem(P) > smem_limit) return false;
    return true;
}

template <typename T>
static cudaError_t set_smem_attrs(const MMParams& P) {
    cudaError_t e;
    if ((e = mm_allow_smem(reinterpret_cast<const void*>(k_fwd_chunk<T>), (int)generic_fwd_smem(P))) != cudaSuccess)
        return e;
    if ((e = mm_allow_smem(reinterpret_cast<const void*>(k_bwd_chunk<T>), (int)generic_bwd_smem(P))) != cudaSuccess)
        return e;
    if ((e = mm_allow_smem(reinterpret_cast<const void*>(k_correct<T>), (int)generic_correct_smem(P))) != cudaSuccess)
        return e;
    return mm_allow_smem(reinterpret_cast<const void*>(k_chunk_end<T>), (int)generic_end_smem(P));
}

template <typename T>
static cudaError_t carries(const MMParams& P, const T* x, const T* bh, const float* da, const float* init,
                           float* Hc, float* Dn, cudaStream_t st) {
    dim3 gch(P.nc, P.h, P.b);
    mm_prof_mark(KID_CHUNK_END, 1, st);
    k_chunk_end<T><<<gch, NT, generic_end_smem(P), st>>>(P, x, bh, da, Hc, Dn);
    mm_prof_mark(KID_CHUNK_END, 0, st);
    return generic_carry_scan(P, init, Hc, Dn, st);
}

template <typename T>
static cudaError_t fwd_impl(const MMParams& P, const GenericPtrs& A, cudaStream_t st) {
    cudaError_t e = set_smem_attrs<T>(P);
    if (e != cudaSuccess) return e;
    const T* x = (const T*)A.xhat;
    const T* bh = (const T*)A.bhat;
    if ((e = carries<T>(P, x, bh, A.da, A.initial, A.Hc, A.Dn, st)) != cudaSuccess) return e;
    dim3 gch(P.nc, P.h, P.b);
    mm_prof_mark(KID_FWD_CHUNK, 1, st);
    k_fwd_chunk<T><<<gch, NT, generic_fwd_smem(P), st>>>(P, x, bh, A.da, A.rot, A.Hc, A.m2, A.m1);
    mm_prof_mark(KID_FWD_CHUNK, 0, st);
    return cudaGetLastError();
}

template <typename T>
static cudaError_t bwd_impl(const MMParams& P, const GenericPtrs& A, int grid, cudaStream_t st) {
    cudaError_t e = set_smem_attrs<T>(P);
    if (e != cudaSuccess) return e;
    const T* x = (const T*)A.xhat;
    const T* bh = (const T*)A.bhat;
    if (!A.reuse_carries && (e = carries<T>(P, x, bh, A.da, A.initial, A.Hc, A.Dn, st)) != cudaSuccess) return e;
    int64_t nbh = (int64_t)P.b * P.h;
    int64_t tot = nbh * P.r * P.r;
    mm_prof_mark(KID_DSYM, 1, st);
    k_dsym<<<(unsigned)((tot + 255) / 256), 256, 0, st>>>(A.dm2, A.dsym, nbh, P.r);
    mm_prof_mark(KID_DSYM, 0, st);
    mm_prof_mark(KID_BWD_CHUNK, 1, st);
    k_bwd_chunk<T><<<grid, NT, generic_bwd_smem(P), st>>>(P, x, bh, A.da, A.rot, A.Hc, A.dsym, A.dm1,
                                                           (T*)A.dxhat, (T*)A.dbhat, A.dda, A.drot,
                                                           A.E, A.traj);
    mm_prof_mark(KID_BWD_CHUNK, 0, st);
    if ((e = generic_cot_scan(P, A.E, A.Dn, A.dinit, st)) != cudaSuccess) return e;
    dim3 gch(P.nc, P.h, P.b);
    mm_prof_mark(KID_CORRECT, 1, st);
    k_correct<T><<<gch, NT, generic_correct_smem(P), st>>>(P, x, bh, A.da, A.Hc, A.E, (T*)A.dxhat,
                                                            (T*)A.dbhat, A.dda);
    mm_prof_mark(KID_CORRECT, 0, st);
    return cudaGetLastError();
}

namespace {
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
template <int V>
dim3 scan_grid(const MMParams& P) {
    const int64_t nv = (int64_t)P.p * P.r / V;
    return dim3((unsigned)((nv + SCAN_T - 1) / SCAN_T), P.h, P.b);
}
}  // namespace

cudaError_t generic_carry_scan(const MMParams& P, const float* initial, float* Hc, const float* Dn,
                               cudaStream_t st) {
    mm_prof_mark(KID_CARRY_SCAN, 1, st);
    if ((P.p * P.r) % 4 == 0 && aligned16(initial) && aligned16(Hc))
        k_carry_scan<4><<<scan_grid<4>(P), SCAN_T, 0, st>>>(P, initial, Hc, Dn);
    else
        k_carry_scan<1><<<scan_grid<1>(P), SCAN_T, 0, st>>>(P, initial, Hc, Dn);
    mm_prof_mark(KID_CARRY_SCAN, 0, st);
    return cudaGetLastError();
}

cudaError_t generic_cot_scan(const MMParams& P, float* E, const float* Dn, float* dinit, cudaStream_t st) {
    mm_prof_mark(KID_COT_SCAN, 1, st);
    if ((P.p * P.r) % 4 == 0 && aligned16(E) && aligned16(dinit))
        k_cot_scan<4><<<scan_grid<4>(P), SCAN_T, 0, st>>>(P, E, Dn, dinit);
    else
        k_cot_scan<1><<<scan_grid<1>(P), SCAN_T, 0, st>>>(P, E, Dn, dinit);
    mm_prof_mark(KID_COT_SCAN, 0, st);
    return cudaGetLastError();
}

cudaError_t generic_dsym(const MMParams& P, const float* dm2, float* dsym, cudaStream_t st) {
    int64_t nbh = (int64_t)P.b * P.h;
    int64_t tot = nbh * P.r * P.r;
    mm_prof_mark(KID_DSYM, 1, st);
    k_dsym<<<(unsigned)((tot + 255) / 256), 256, 0, st>>>(dm2, dsym, nbh, P.r);
    mm_prof_mark(KID_DSYM, 0, st);
    return cudaGetLastError();
}

cudaError_t generic_fwd(const MMParams& P, bool bf16, const GenericPtrs& A, cudaStream_t st) {
    return bf16 ? fwd_impl<__nv_bfloat16>(P, A, st) : fwd_impl<float>(P, A, st);
}
cudaError_t generic_bwd(const MMParams& P, bool bf16, const GenericPtrs& A, int grid, cudaStream_t st) {
    return bf16 ? bwd_impl<__nv_bfloat16>(P, A, grid, st) : bwd_impl<float>(P, A, grid, st);
}
