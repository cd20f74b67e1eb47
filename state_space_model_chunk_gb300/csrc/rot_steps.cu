// rot_steps.cu -- the per-token cumulative rotation built from per-token steps, and the gradient
// of that build, for calls made with MM_FLAG_ROT_STEPS.
//
// The operator consumes the cumulative rotation of every token ("mamba3/moments/recalculated.rs",
// RotPrim: cumulative angles [b, s, h, a] or cumulative unit quaternions [b, s, h, J, 4]); its
// producer (RotationSeq, rotation::quat_mul) is named there but not given.  Built here as:
//   angles       theta_t = sum_{u <= t} dtheta_u                       (inclusive prefix sum)
//   quaternions  Q_t = q_t (x) Q_{t-1},  Q_{-1} = 1                     (running Hamilton product)
// and, in reverse mode,
//   angles       d_dtheta_u = sum_{t >= u} d_theta_t
//   quaternions  G_t = dQ_t + conj(q_{t+1}) (x) G_{t+1},  d_q_t = G_t (x) conj(Q_{t-1}).
//
// Each is a scan along the sequence, done in three passes over 64-token chunks so that every pass
// is parallel over (batch row, chunk, head x angle): (1) a summary per chunk (a sum; a product of
// the chunk's steps; for the quaternion gradient the carry the chunk passes on with nothing coming
// in, and the product of its conjugated steps that maps an incoming carry through it), (2) a scan
// of the summaries over the chunks of a row, (3) the chunk again from its incoming value.  Threads
// own one (head, angle) column or one (head, block) quaternion; the loads of a token are contiguous
// across threads.
#include "prof.h"
#include "rot_steps.h"

namespace {

constexpr int TCH = 64;   // tokens per chunk of the scans
constexpr int NTH = 256;  // threads per block

__device__ __forceinline__ float4 qmul(const float4 a, const float4 b) {
    return make_float4(a.x * b.x - a.y * b.y - a.z * b.z - a.w * b.w, a.x * b.y + a.y * b.x + a.z * b.w - a.w * b.z,
                       a.x * b.z - a.y * b.w + a.z * b.x + a.w * b.y, a.x * b.w + a.y * b.z - a.z * b.y + a.w * b.x);
}
__device__ __forceinline__ float4 qconj(const float4 q) { return make_float4(q.x, -q.y, -q.z, -q.w); }
__device__ __forceinline__ float4 qadd(const float4 a, const float4 b) {
    return make_float4(a.x + b.x, a.y + b.y, a.z + b.z, a.w + b.w);
}

struct Geo {
    int b, s, nck;
    int ncol;  // columns per token: h * a floats (angles) or h * J quaternions
};

// ------------------------------------------------------------------------------- angle steps
// x [b, s, ncol] -> tot [b, nck, ncol]: the sum of each chunk
__global__ void __launch_bounds__(NTH) k_ang_sum(Geo g, const float* __restrict__ x, float* __restrict__ tot) {
    const int col = blockIdx.x * NTH + threadIdx.x, ck = blockIdx.y, bb = blockIdx.z;
    if (col >= g.ncol) return;
    const int t0 = ck * TCH, t1 = min(g.s, t0 + TCH);
    const float* p = x + ((int64_t)bb * g.s + t0) * g.ncol + col;
    float acc = 0.f;
#pragma unroll 8
    for (int t = t0; t < t1; ++t, p += g.ncol) acc += *p;
    tot[((int64_t)bb * g.nck + ck) * g.ncol + col] = acc;
}
// in place: chunk sums -> the sum of every earlier chunk (rev: of every later chunk)
__global__ void __launch_bounds__(NTH) k_ang_scan(Geo g, float* __restrict__ tot, int rev) {
    const int col = blockIdx.x * NTH + threadIdx.x, bb = blockIdx.y;
    if (col >= g.ncol) return;
    float* p = tot + (int64_t)bb * g.nck * g.ncol + col;
    float run = 0.f;
    for (int i = 0; i < g.nck; ++i) {
        const int ck = rev ? g.nck - 1 - i : i;
        const float v = p[(int64_t)ck * g.ncol];
        p[(int64_t)ck * g.ncol] = run;
        run += v;
    }
}
// y[t] = offset of the chunk + the sum of the chunk's x up to t (rev: from t to the chunk's end)
__global__ void __launch_bounds__(NTH) k_ang_apply(Geo g, const float* __restrict__ x, const float* __restrict__ off,
                                                   float* __restrict__ y, int rev) {
    const int col = blockIdx.x * NTH + threadIdx.x, ck = blockIdx.y, bb = blockIdx.z;
    if (col >= g.ncol) return;
    const int t0 = ck * TCH, t1 = min(g.s, t0 + TCH);
    float run = off[((int64_t)bb * g.nck + ck) * g.ncol + col];
    const int64_t base = (int64_t)bb * g.s * g.ncol + col;
    if (!rev) {
        for (int t = t0; t < t1; ++t) {
            run += x[base + (int64_t)t * g.ncol];
            y[base + (int64_t)t * g.ncol] = run;
        }
    } else {
        for (int t = t1 - 1; t >= t0; --t) {
            run += x[base + (int64_t)t * g.ncol];
            y[base + (int64_t)t * g.ncol] = run;
        }
    }
}

// -------------------------------------------------------------------------- quaternion steps
// q [b, s, ncol] float4 -> P [b, nck, ncol]: q_last (x) ... (x) q_first of each chunk
__global__ void __launch_bounds__(NTH) k_quat_prod(Geo g, const float4* __restrict__ q, float4* __restrict__ P) {
    const int col = blockIdx.x * NTH + threadIdx.x, ck = blockIdx.y, bb = blockIdx.z;
    if (col >= g.ncol) return;
    const int t0 = ck * TCH, t1 = min(g.s, t0 + TCH);
    const float4* p = q + ((int64_t)bb * g.s + t0) * g.ncol + col;
    float4 acc = make_float4(1.f, 0.f, 0.f, 0.f);
    for (int t = t0; t < t1; ++t, p += g.ncol) acc = qmul(*p, acc);
    P[((int64_t)bb * g.nck + ck) * g.ncol + col] = acc;
}
// in place: chunk products -> the rotation accumulated before each chunk
__global__ void __launch_bounds__(NTH) k_quat_scan(Geo g, float4* __restrict__ P) {
    const int col = blockIdx.x * NTH + threadIdx.x, bb = blockIdx.y;
    if (col >= g.ncol) return;
    float4* p = P + (int64_t)bb * g.nck * g.ncol + col;
    float4 run = make_float4(1.f, 0.f, 0.f, 0.f);
    for (int ck = 0; ck < g.nck; ++ck) {
        const float4 v = p[(int64_t)ck * g.ncol];
        p[(int64_t)ck * g.ncol] = run;
        run = qmul(v, run);
    }
}
__global__ void __launch_bounds__(NTH) k_quat_apply(Geo g, const float4* __restrict__ q, const float4* __restrict__ Pin,
                                                    float4* __restrict__ Q) {
    const int col = blockIdx.x * NTH + threadIdx.x, ck = blockIdx.y, bb = blockIdx.z;
    if (col >= g.ncol) return;
    const int t0 = ck * TCH, t1 = min(g.s, t0 + TCH);
    float4 run = Pin[((int64_t)bb * g.nck + ck) * g.ncol + col];
    const int64_t base = (int64_t)bb * g.s * g.ncol + col;
    for (int t = t0; t < t1; ++t) {
        run = qmul(q[base + (int64_t)t * g.ncol], run);
        Q[base + (int64_t)t * g.ncol] = run;
    }
}

// gradient, pass 1: per chunk, the carry it passes to the token before it with nothing coming in
// from after it (H), and K = conj(q_first) (x) ... (x) conj(q_last), which maps an incoming carry
// through the chunk: S[b, nck, ncol][2] = {H, K}
__global__ void __launch_bounds__(NTH) k_quatg_chunk(Geo g, const float4* __restrict__ q, const float4* __restrict__ dQ,
                                                     float4* __restrict__ S) {
    const int col = blockIdx.x * NTH + threadIdx.x, ck = blockIdx.y, bb = blockIdx.z;
    if (col >= g.ncol) return;
    const int t0 = ck * TCH, t1 = min(g.s, t0 + TCH);
    const int64_t base = (int64_t)bb * g.s * g.ncol + col;
    float4 H = make_float4(0.f, 0.f, 0.f, 0.f), K = make_float4(1.f, 0.f, 0.f, 0.f);
    for (int t = t1 - 1; t >= t0; --t) {
        const float4 cq = qconj(q[base + (int64_t)t * g.ncol]);
        H = qmul(cq, qadd(dQ[base + (int64_t)t * g.ncol], H));
        K = qmul(cq, K);
    }
    float4* o = S + (((int64_t)bb * g.nck + ck) * g.ncol + col) * 2;
    o[0] = H;
    o[1] = K;
}
// pass 2: from the last chunk back, the carry coming into each chunk from the chunks after it
// (stored over the chunk's H)
__global__ void __launch_bounds__(NTH) k_quatg_scan(Geo g, float4* __restrict__ S) {
    const int col = blockIdx.x * NTH + threadIdx.x, bb = blockIdx.y;
    if (col >= g.ncol) return;
    float4 in = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int ck = g.nck - 1; ck >= 0; --ck) {
        float4* o = S + (((int64_t)bb * g.nck + ck) * g.ncol + col) * 2;
        const float4 H = o[0], K = o[1];
        o[0] = in;
        in = qadd(H, qmul(K, in));
    }
}
// pass 3: the chunk again from its incoming carry: G_t = dQ_t + carry, d_q_t = G_t (x) conj(Q_{t-1})
__global__ void __launch_bounds__(NTH) k_quatg_apply(Geo g, const float4* __restrict__ q, const float4* __restrict__ Q,
                                                     const float4* __restrict__ dQ, const float4* __restrict__ S,
                                                     float4* __restrict__ dq) {
    const int col = blockIdx.x * NTH + threadIdx.x, ck = blockIdx.y, bb = blockIdx.z;
    if (col >= g.ncol) return;
    const int t0 = ck * TCH, t1 = min(g.s, t0 + TCH);
    const int64_t base = (int64_t)bb * g.s * g.ncol + col;
    float4 H = S[(((int64_t)bb * g.nck + ck) * g.ncol + col) * 2];
    for (int t = t1 - 1; t >= t0; --t) {
        const int64_t i = base + (int64_t)t * g.ncol;
        const float4 G = qadd(dQ[i], H);
        const float4 prev = t > 0 ? Q[i - g.ncol] : make_float4(1.f, 0.f, 0.f, 0.f);
        dq[i] = qmul(G, qconj(prev));
        H = qmul(qconj(q[i]), G);
    }
}

// each launch between its own pair of profiling marks
#define MARKED(...)                         \
    do {                                    \
        mm_prof_mark(KID_ROT_STEPS, 1, st); \
        __VA_ARGS__;                        \
        mm_prof_mark(KID_ROT_STEPS, 0, st); \
    } while (0)

Geo geo_of(const MMParams& P) {
    Geo g;
    g.b = P.b;
    g.s = P.s;
    g.nck = (P.s + TCH - 1) / TCH;
    g.ncol = P.h * (P.rot == ROT_QUAT ? P.J : P.na);
    return g;
}

}  // namespace

size_t rot_steps_scratch_bytes(const MMParams& P) {
    const Geo g = geo_of(P);
    // angles: one float per (row, chunk, column); quaternions: two float4 (the gradient's pass)
    const size_t per = P.rot == ROT_QUAT ? 2 * sizeof(float4) : sizeof(float);
    return (size_t)g.b * g.nck * g.ncol * per;
}

cudaError_t rot_steps_build(const MMParams& P, const float* steps, float* cum, void* scratch, cudaStream_t st) {
    const Geo g = geo_of(P);
    if (g.ncol == 0) return cudaSuccess;
    if (g.nck > 65535) return cudaErrorInvalidValue;  // chunks go in grid.y
    const dim3 grid3((g.ncol + NTH - 1) / NTH, g.nck, g.b), grid2((g.ncol + NTH - 1) / NTH, g.b);
    if (P.rot == ROT_QUAT) {
        float4* S = static_cast<float4*>(scratch);
        MARKED(k_quat_prod<<<grid3, NTH, 0, st>>>(g, reinterpret_cast<const float4*>(steps), S));
        MARKED(k_quat_scan<<<grid2, NTH, 0, st>>>(g, S));
        MARKED(k_quat_apply<<<grid3, NTH, 0, st>>>(g, reinterpret_cast<const float4*>(steps), S, reinterpret_cast<float4*>(cum)));
    } else {
        float* S = static_cast<float*>(scratch);
        MARKED(k_ang_sum<<<grid3, NTH, 0, st>>>(g, steps, S));
        MARKED(k_ang_scan<<<grid2, NTH, 0, st>>>(g, S, 0));
        MARKED(k_ang_apply<<<grid3, NTH, 0, st>>>(g, steps, S, cum, 0));
    }
    return cudaGetLastError();
}

cudaError_t rot_steps_vjp(const MMParams& P, const float* steps, const float* cum, const float* d_cum, float* d_steps,
                          void* scratch, cudaStream_t st) {
    const Geo g = geo_of(P);
    if (g.ncol == 0) return cudaSuccess;
    if (g.nck > 65535) return cudaErrorInvalidValue;
    const dim3 grid3((g.ncol + NTH - 1) / NTH, g.nck, g.b), grid2((g.ncol + NTH - 1) / NTH, g.b);
    if (P.rot == ROT_QUAT) {
        const float4* q = reinterpret_cast<const float4*>(steps);
        const float4* dQ = reinterpret_cast<const float4*>(d_cum);
        float4* S = static_cast<float4*>(scratch);
        MARKED(k_quatg_chunk<<<grid3, NTH, 0, st>>>(g, q, dQ, S));
        MARKED(k_quatg_scan<<<grid2, NTH, 0, st>>>(g, S));
        MARKED(k_quatg_apply<<<grid3, NTH, 0, st>>>(g, q, reinterpret_cast<const float4*>(cum), dQ, S,
                                             reinterpret_cast<float4*>(d_steps)));
    } else {
        float* S = static_cast<float*>(scratch);
        MARKED(k_ang_sum<<<grid3, NTH, 0, st>>>(g, d_cum, S));
        MARKED(k_ang_scan<<<grid2, NTH, 0, st>>>(g, S, 1));
        MARKED(k_ang_apply<<<grid3, NTH, 0, st>>>(g, d_cum, S, d_steps, 1));
    }
    return cudaGetLastError();
}
