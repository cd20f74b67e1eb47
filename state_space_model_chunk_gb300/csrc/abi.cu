// abi.cu -- the extern "C" boundary of libmoments.so: validation, workspace layout, dispatch.
// Declarations and the full contract: include/moments.h.
#include <cstring>
#include <mutex>
#include <vector>

#include "../../include/moments.h"
#include "common.cuh"
#include "fast.h"
#include "finite.h"
#include "generic.h"
#include "noalloc.h"
#include "prof.h"
#include "rot_steps.h"

namespace {

constexpr size_t kAlign = 256;
constexpr int kTrajSlots = 320;  // blocks of the SIMT backward (>= 2 per SM on 152 SMs)
constexpr size_t kHeader = 256;  // workspace header: status words (timeout at offset 0, non-finite at 4)

size_t align_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

struct Layout {
    size_t Hc = 0, Dn = 0, E = 0, dsym = 0, traj = 0, fast = 0, total = 0;
    size_t cum = 0, dcum = 0, rsc = 0;  // MM_FLAG_ROT_STEPS: cumulative rotation, its gradient, scan scratch
    bool steps = false;
};

bool valid_problem(const mm_problem* P) {
    if (!P) return false;
    if (P->b < 1 || P->s < 1 || P->C < 1 || P->h < 1 || P->p < 1 || P->r < 1 || P->chunk_len < 1) return false;
    if (P->s % P->chunk_len) return false;
    if (P->xb_dtype != MM_F32 && P->xb_dtype != MM_BF16) return false;
    switch (P->rot) {
        case MM_ROT_NONE: break;
        case MM_ROT_PAIRWISE:
            if (P->rope_dim < 0 || P->rope_dim % 2 || P->rope_dim > P->r) return false;
            break;
        case MM_ROT_HALF:
            if (P->rope_dim < 0 || P->rope_dim % 2 || P->r % 2 || P->rope_dim / 2 > P->r / 2) return false;
            break;
        case MM_ROT_QUAT:
            if (P->quat_blocks < 0 || 4 * P->quat_blocks > P->r) return false;
            break;
        default: return false;
    }
    // sizes the kernels index with 32-bit block coordinates
    if (P->h > 65535 || P->b > 65535 || P->s / P->chunk_len > (int64_t)1 << 30) return false;
    if (P->p > 4096 || P->r > 4096 || P->C > 4096 || P->chunk_len > 65536 || P->s > ((int64_t)1 << 31) - 1)
        return false;
    return true;
}

int rot_width(const mm_problem* P) {
    if (P->rot == MM_ROT_PAIRWISE || P->rot == MM_ROT_HALF) return (int)(P->rope_dim / 2);
    if (P->rot == MM_ROT_QUAT) return (int)(4 * P->quat_blocks);
    return 0;
}

void fill_params(const mm_problem* P, const int64_t* valid_host, MMParams* out) {
    std::memset(out, 0, sizeof(*out));
    out->b = (int)P->b; out->s = (int)P->s; out->C = (int)P->C; out->h = (int)P->h;
    out->p = (int)P->p; out->r = (int)P->r; out->l = (int)P->chunk_len;
    out->nc = (int)(P->s / P->chunk_len);
    out->rot = P->rot;
    out->na = (P->rot == MM_ROT_PAIRWISE || P->rot == MM_ROT_HALF) ? (int)(P->rope_dim / 2) : 0;
    out->J = (P->rot == MM_ROT_QUAT) ? (int)P->quat_blocks : 0;
    out->rw = rot_width(P);
    out->heads = out->h;
    out->groups = 1;
    out->prow = out->p;
    for (int64_t i = 0; i < P->b && valid_host; ++i) {
        int64_t v = valid_host[i];
        out->valid[i] = (int)(v < 0 ? 0 : (v > P->s ? P->s : v));
    }
}

int smem_optin_limit() {
    int dev = 0, v = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) { cudaGetLastError(); return 232448; }
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess) {
        cudaGetLastError();
        return 232448;
    }
    return v;
}

bool use_fast(const mm_problem* P, const MMParams& M, int backward) {
    if (P->flags & MM_FLAG_FORCE_GENERIC) return false;
    return fast_supported(M, P->xb_dtype == MM_BF16, backward);
}

Layout layout(const mm_problem* P, int backward) {
    Layout L;
    MMParams M;
    fill_params(P, nullptr, &M);
    const bool fast = use_fast(P, M, backward);
    // the tensor-core path keeps its carries at a fixed 64-token granularity
    const size_t l_eff = fast ? (size_t)fastk_chunk() : (size_t)P->chunk_len;
    // (the tensor-core path runs at least 64 state rows per head: p below 64 is padded with zero rows)
    const size_t pr = (size_t)((fast && P->p < 64) ? 64 : P->p) * P->r;
    const size_t nbh = (size_t)P->b * P->h;
    const size_t nc = ((size_t)P->s + l_eff - 1) / l_eff;  // (the tensor-core path's last chunk may be partial)
    size_t off = kHeader;  // header: device error word
    L.Hc = off; off = align_up(off + sizeof(float) * nbh * nc * pr);
    // chunk decays: per head, or on the tensor-core path per 64-row group of a head (each group
    // runs as a head of its own)
    const size_t groups = (fast && P->p > 64) ? (size_t)P->p / 64 : 1;
    L.Dn = off; off = align_up(off + sizeof(float) * nbh * groups * nc);
    // MM_FLAG_ROT_STEPS: the cumulative rotation sits right after the carries, at the same offset
    // in the forward's and the backward's layout, so a backward reusing the forward's carries
    // reuses it too
    L.steps = (P->flags & MM_FLAG_ROT_STEPS) && M.rw > 0;
    const size_t nrot = sizeof(float) * (size_t)P->b * P->s * P->h * M.rw;
    if (L.steps) { L.cum = off; off = align_up(off + nrot); }
    if (backward) {
        L.E = off; off = align_up(off + sizeof(float) * nbh * nc * pr);
        L.dsym = off; off = align_up(off + sizeof(float) * nbh * (size_t)P->r * P->r);
    }
    if (fast) {
        L.fast = off; off = align_up(off + fast_scratch_bytes(M, backward));
    } else if (backward) {
        L.traj = off; off = align_up(off + sizeof(float) * (size_t)kTrajSlots * P->chunk_len * pr);
    }
    if (L.steps) {
        if (backward) { L.dcum = off; off = align_up(off + nrot); }
        L.rsc = off; off = align_up(off + rot_steps_scratch_bytes(M));
    }
    L.total = off;
    if (backward) {
        // a backward-sized workspace also serves the forward (MM_FLAG_REUSE_CARRIES hands one
        // workspace to both calls)
        const size_t fwd_total = layout(P, 0).total;
        if (fwd_total > L.total) L.total = fwd_total;
    }
    return L;
}

template <typename T>
T* at(void* base, size_t off) { return reinterpret_cast<T*>(static_cast<char*>(base) + off); }

// Tensor pointers must start on a 16-byte boundary (the kernels move 16-byte vectors and tensor
// copies); NULL passes (presence is checked separately).
bool misaligned(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) != 0; }

mm_status common_checks(const mm_problem* P, const void* xhat, const void* bhat, const float* da,
                        const float* rot, const float* initial, const int64_t* valid, void* ws,
                        size_t ws_bytes, int backward, Layout* L) {
    if (!valid_problem(P)) return MM_ERR_INVALID_ARG;
    if (!xhat || !bhat || !da || !initial || !valid) return MM_ERR_INVALID_ARG;
    if (rot_width(P) > 0 && !rot) return MM_ERR_INVALID_ARG;
    if (misaligned(xhat) || misaligned(bhat) || misaligned(da) || misaligned(rot) || misaligned(initial))
        return MM_ERR_INVALID_ARG;
    for (int64_t i = 0; i < P->b; ++i)
        if (valid[i] < 0) return MM_ERR_INVALID_ARG;
    if (P->b > MM_MAX_B) return MM_ERR_UNSUPPORTED;
    *L = layout(P, backward);
    if (!ws || (reinterpret_cast<uintptr_t>(ws) % kAlign) || ws_bytes < L->total) return MM_ERR_WORKSPACE;
    return MM_OK;
}

}  // namespace

// ------------------------------------------------------------------ optional profiling
namespace {
struct ProfRec { int kid; cudaEvent_t a, b; };
std::mutex g_prof_mu;
bool g_prof_on = false;
std::vector<ProfRec> g_recs;
std::vector<cudaEvent_t> g_pool;
int g_open[KID_COUNT];
cudaEvent_t take_event() {
    if (!g_pool.empty()) { cudaEvent_t e = g_pool.back(); g_pool.pop_back(); return e; }
    cudaEvent_t e = nullptr;
    if (cudaEventCreate(&e) != cudaSuccess) { cudaGetLastError(); return nullptr; }
    return e;
}
const char* kKernelNames[KID_COUNT] = {
    "chunk_end", "carry_scan", "fwd_chunk", "dsym", "bwd_chunk", "cot_scan", "correct",
    "tc_fwd_chunk", "tc_chunk_end", "tc_bwd_chunk", "tc_correct", "check_finite", "m2_reduce", "drot_sum", "rot_steps",
    "group_sum"};
}  // namespace

void mm_prof_mark(int kid, int begin, cudaStream_t st) {
    if (!g_prof_on) return;
    std::lock_guard<std::mutex> g(g_prof_mu);
    cudaEvent_t e = take_event();
    if (!e) return;
    cudaEventRecord(e, st);
    if (begin) {
        g_recs.push_back(ProfRec{kid, e, nullptr});
        g_open[kid] = (int)g_recs.size() - 1;
    } else if (g_open[kid] >= 0) {
        g_recs[g_open[kid]].b = e;
        g_open[kid] = -1;
    } else {
        g_pool.push_back(e);
    }
}

cudaError_t mm_allow_smem(const void* fn, int bytes) {
    static std::mutex mu;
    static std::vector<std::pair<std::pair<const void*, int>, int>> done;  // (function, device) -> bytes
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> g(mu);
    for (auto& d : done)
        if (d.first.first == fn && d.first.second == dev) {
            if (d.second >= bytes) return cudaSuccess;
            if ((e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes)) == cudaSuccess)
                d.second = bytes;
            return e;
        }
    if ((e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes)) == cudaSuccess)
        done.push_back({{fn, dev}, bytes});
    return e;
}

extern "C" {

size_t mm_workspace_bytes(const mm_problem* prob, int backward) {
    if (!valid_problem(prob)) return 0;
    return layout(prob, backward).total;
}

int mm_path(const mm_problem* prob, int backward) {
    if (!valid_problem(prob)) return -1;
    MMParams M;
    fill_params(prob, nullptr, &M);
    return use_fast(prob, M, backward) ? 1 : 0;
}

void mm_profile_enable(int on) {
    std::lock_guard<std::mutex> g(g_prof_mu);
    if (!on) { g_prof_on = false; return; }  // stop recording, keep the records for collection
    for (auto& r : g_recs) {
        if (r.a) g_pool.push_back(r.a);
        if (r.b) g_pool.push_back(r.b);
    }
    g_recs.clear();
    for (int i = 0; i < KID_COUNT; ++i) g_open[i] = -1;
    g_prof_on = true;
}

int mm_profile_collect(double* total_ms, int64_t* launches, int n) {
    std::lock_guard<std::mutex> g(g_prof_mu);
    for (int i = 0; i < n && i < KID_COUNT; ++i) { total_ms[i] = 0.0; launches[i] = 0; }
    for (auto& r : g_recs) {
        if (!r.a || !r.b || r.kid >= n) continue;
        if (cudaEventSynchronize(r.b) != cudaSuccess) { cudaGetLastError(); return -1; }
        float ms = 0.f;
        if (cudaEventElapsedTime(&ms, r.a, r.b) != cudaSuccess) { cudaGetLastError(); return -1; }
        total_ms[r.kid] += ms;
        launches[r.kid] += 1;
    }
    return KID_COUNT;
}

const char* mm_kernel_name(int id) { return (id >= 0 && id < KID_COUNT) ? kKernelNames[id] : "?"; }

mm_status mm_device_status(const void* workspace, void* stream) {
    if (!workspace) {  // the fixed scratch of moments_fwd_noalloc on the current device
        void* p = nullptr;
        const mm_status st = noalloc_scratch(stream, &p);
        if (st != MM_OK) return st;
        workspace = p;
    }
    int v[2] = {0, 0};  // [0]: a bounded device wait gave up; [1]: the finiteness check fired
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    if (cudaMemcpyAsync(v, workspace, sizeof(v), cudaMemcpyDeviceToHost, cs) != cudaSuccess ||
        cudaStreamSynchronize(cs) != cudaSuccess) {
        cudaGetLastError();
        return MM_ERR_CUDA;
    }
    if (v[0]) return MM_ERR_TIMEOUT;
    if (v[1]) return MM_ERR_NONFINITE;
    return MM_OK;
}

const char* mm_status_string(mm_status s) {
    switch (s) {
        case MM_OK: return "ok";
        case MM_ERR_INVALID_ARG: return "invalid argument";
        case MM_ERR_UNSUPPORTED: return "unsupported problem for this build";
        case MM_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
        case MM_ERR_CUDA: return "CUDA launch error";
        case MM_ERR_NONFINITE: return "non-finite values detected";
        case MM_ERR_TIMEOUT: return "device-side wait timed out";
    }
    return "unknown status";
}

mm_status moments_fwd(const mm_problem* prob, const void* xhat, const void* bhat, const float* da,
                      const float* rot, const float* initial, const int64_t* valid_len_host, float* m2,
                      float* m1, void* workspace, size_t ws_bytes, void* stream) {
    Layout L;
    mm_status st = common_checks(prob, xhat, bhat, da, rot, initial, valid_len_host, workspace, ws_bytes, 0, &L);
    if (st != MM_OK) return st;
    if (!m2 || !m1 || misaligned(m2) || misaligned(m1)) return MM_ERR_INVALID_ARG;
    MMParams M;
    fill_params(prob, valid_len_host, &M);
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    const bool bf16 = prob->xb_dtype == MM_BF16;
    const bool fast = use_fast(prob, M, 0);
    if (!fast && !generic_supported(M, smem_optin_limit())) return MM_ERR_UNSUPPORTED;
    const size_t nbh = (size_t)prob->b * prob->h;
    if (cudaMemsetAsync(m2, 0, sizeof(float) * nbh * prob->r * prob->r, cs) != cudaSuccess ||
        cudaMemsetAsync(m1, 0, sizeof(float) * nbh * prob->r, cs) != cudaSuccess) {
        cudaGetLastError();
        return MM_ERR_CUDA;
    }
    GenericPtrs A{};
    A.xhat = xhat; A.bhat = bhat; A.da = da; A.rot = rot; A.initial = initial; A.m2 = m2; A.m1 = m1;
    A.Hc = at<float>(workspace, L.Hc);
    A.Dn = at<float>(workspace, L.Dn);
    A.test_wait_timeout = (prob->flags & MM_FLAG_TEST_WAIT_TIMEOUT) ? 1 : 0;
    A.err = at<int>(workspace, 0);
    if (cudaMemsetAsync(A.err, 0, 2 * sizeof(int), cs) != cudaSuccess) { cudaGetLastError(); return MM_ERR_CUDA; }
    cudaError_t e = cudaSuccess;
    if (L.steps) {  // the operator runs on the cumulative rotation built from the steps
        e = rot_steps_build(M, rot, at<float>(workspace, L.cum), at<void>(workspace, L.rsc), cs);
        A.rot = at<float>(workspace, L.cum);
    }
    if (e == cudaSuccess) e = fast ? fast_fwd(M, A, at<char>(workspace, L.fast), cs) : generic_fwd(M, bf16, A, cs);
    if (e == cudaSuccess && (prob->flags & MM_FLAG_CHECK_FINITE)) {
        FiniteSegs fs{};
        fs.n = 2;
        fs.ptr[0] = m2; fs.bytes[0] = (int64_t)(sizeof(float) * nbh * prob->r * prob->r);
        fs.ptr[1] = m1; fs.bytes[1] = (int64_t)(sizeof(float) * nbh * prob->r);
        e = launch_finite_check(fs, at<int>(workspace, 4), cs);
    }
    if (e != cudaSuccess) { cudaGetLastError(); return MM_ERR_CUDA; }
    return MM_OK;
}

mm_status moments_bwd(const mm_problem* prob, const void* xhat, const void* bhat, const float* da,
                      const float* rot, const float* initial, const int64_t* valid_len_host,
                      const float* d_m2, const float* d_m1, void* d_xhat, void* d_bhat, float* d_da,
                      float* d_rot, float* d_initial, void* workspace, size_t ws_bytes, void* stream) {
    Layout L;
    mm_status st = common_checks(prob, xhat, bhat, da, rot, initial, valid_len_host, workspace, ws_bytes, 1, &L);
    if (st != MM_OK) return st;
    if (!d_m2 || !d_m1 || !d_xhat || !d_bhat || !d_da || !d_initial) return MM_ERR_INVALID_ARG;
    if (rot_width(prob) > 0 && !d_rot) return MM_ERR_INVALID_ARG;
    if (misaligned(d_m2) || misaligned(d_m1) || misaligned(d_xhat) || misaligned(d_bhat) || misaligned(d_da) ||
        misaligned(d_rot) || misaligned(d_initial))
        return MM_ERR_INVALID_ARG;
    MMParams M;
    fill_params(prob, valid_len_host, &M);
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    const bool bf16 = prob->xb_dtype == MM_BF16;
    const bool fast = use_fast(prob, M, 1);
    if (!fast && !generic_supported(M, smem_optin_limit())) return MM_ERR_UNSUPPORTED;
    const size_t es = bf16 ? 2 : 4;
    const size_t ntok = (size_t)prob->b * prob->s;
    const size_t nx = ntok * prob->C * prob->h * prob->p, nb = ntok * prob->C * prob->h * prob->r;
    const size_t nrot = ntok * prob->h * (size_t)rot_width(prob);
    GenericPtrs A{};
    A.xhat = xhat; A.bhat = bhat; A.da = da; A.rot = rot; A.initial = initial;
    A.dm2 = d_m2; A.dm1 = d_m1; A.dxhat = d_xhat; A.dbhat = d_bhat; A.dda = d_da; A.drot = d_rot;
    A.dinit = d_initial;
    // carries from the forward: only where both directions share the path (and so the layout)
    A.reuse_carries = (prob->flags & MM_FLAG_REUSE_CARRIES) && use_fast(prob, M, 0) == fast;
    A.Hc = at<float>(workspace, L.Hc);
    A.Dn = at<float>(workspace, L.Dn);
    A.E = at<float>(workspace, L.E);
    A.dsym = at<float>(workspace, L.dsym);
    A.err = at<int>(workspace, 0);
    if (cudaMemsetAsync(A.err, 0, 2 * sizeof(int), cs) != cudaSuccess) { cudaGetLastError(); return MM_ERR_CUDA; }
    cudaError_t e = cudaSuccess;
    if (L.steps) {  // the operator's gradient w.r.t. the cumulative rotation goes to the workspace
        // (the forward of the same problem left the cumulative rotation where the carries are)
        if (!A.reuse_carries) e = rot_steps_build(M, rot, at<float>(workspace, L.cum), at<void>(workspace, L.rsc), cs);
        A.rot = at<float>(workspace, L.cum);
        A.drot = at<float>(workspace, L.dcum);
    }
    if (e != cudaSuccess) {
    } else if (fast) {
        e = fast_bwd(M, A, at<char>(workspace, L.fast), cs);
    } else {
        // every gradient position not written by a kernel must read zero
        if (cudaMemsetAsync(d_xhat, 0, es * nx, cs) != cudaSuccess ||
            cudaMemsetAsync(d_bhat, 0, es * nb, cs) != cudaSuccess ||
            cudaMemsetAsync(d_da, 0, sizeof(float) * ntok * prob->h, cs) != cudaSuccess ||
            (nrot && cudaMemsetAsync(A.drot, 0, sizeof(float) * nrot, cs) != cudaSuccess)) {
            cudaGetLastError();
            return MM_ERR_CUDA;
        }
        A.traj = at<float>(workspace, L.traj);
        int64_t chunks = (int64_t)prob->b * prob->h * (prob->s / prob->chunk_len);
        int grid = (int)(chunks < kTrajSlots ? chunks : kTrajSlots);
        e = generic_bwd(M, bf16, A, grid, cs);
    }
    if (e == cudaSuccess && L.steps)  // through the build: the gradient w.r.t. the steps
        e = rot_steps_vjp(M, rot, A.rot, A.drot, d_rot, at<void>(workspace, L.rsc), cs);
    if (e == cudaSuccess && (prob->flags & MM_FLAG_CHECK_FINITE)) {
        FiniteSegs fs{};
        const void* outs[5] = {d_xhat, d_bhat, d_da, d_rot, d_initial};
        const size_t nbytes[5] = {es * nx, es * nb, sizeof(float) * ntok * prob->h, sizeof(float) * nrot,
                                  sizeof(float) * (size_t)prob->b * prob->h * prob->p * prob->r};
        for (int i = 0; i < 5; ++i) {
            if (!outs[i] || !nbytes[i]) continue;
            fs.ptr[fs.n] = outs[i];
            fs.bytes[fs.n] = (int64_t)nbytes[i];
            fs.bf16[fs.n] = (i < 2 && bf16) ? 1 : 0;
            ++fs.n;
        }
        e = launch_finite_check(fs, at<int>(workspace, 4), cs);
    }
    if (e != cudaSuccess) { cudaGetLastError(); return MM_ERR_CUDA; }
    return MM_OK;
}

}  // extern "C"
