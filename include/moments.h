/*
 * moments.h -- C ABI of libmoments.so, the GB300 (sm_103a) physical-frame state-moments
 * operator and its recompute backward.
 *
 * The operation (burn-mamba, "mamba3/moments/recalculated.rs", trait
 * Mamba3MomentsBackendExt::mamba3_state_moments_phys and moments_phys_fwd; backward in
 * "mamba3/moments/backward.rs", moments_phys_bwd and its module header "Gradient math"):
 *
 *   per batch row b and head h, with a_t the cumulative da and h_{-1} = initial[b,h]:
 *     h_t = exp(da[b,t,h]) h_{t-1} + sum_c xhat[b,t,c,h,:] (x) bhat[b,t,c,h,:]      (p x r)
 *     c_t = derot_t(h_t)          on the r axis of every row: complex pairs by R(-theta)
 *                                 (pairwise (2i,2i+1) or half-split (i, i+r/2)), or each
 *                                 4-block left-multiplied by the unit quaternion Q
 *     m2[b,h] = sum_{t < valid_len[b]} sum_p c_t[p,:]^T c_t[p,:]     [r, r]   (raw sum)
 *     m1[b,h] = sum_{t < valid_len[b]} sum_p c_t[p,:]                [r]
 *   The backward returns the gradients of <d_m2, m2> + <d_m1, m1> with respect to all five
 *   inputs.  The state trajectory is never written to memory: chunk-boundary carries are
 *   computed by a cheap chunk-level pass and each chunk is recomputed on chip.
 *
 * Conventions
 *   - Every tensor is dense row-major (C order) with exactly the shapes given below.
 *     xhat [b,s,C,h,p], bhat [b,s,C,h,r]: element type mm_problem.xb_dtype (fp32 or bf16).
 *     da [b,s,h], initial [b,h,p,r], m2/d_m2 [b,h,r,r], m1/d_m1 [b,h,r]: fp32.
 *     rot: fp32 [b,s,h,rope_dim/2] cumulative angles (MM_ROT_PAIRWISE / MM_ROT_HALF) or
 *          [b,s,h,quat_blocks,4] cumulative quaternions (w,x,y,z) (MM_ROT_QUAT); may be
 *          NULL when there is nothing to rotate (MM_ROT_NONE, rope_dim 0 or 0 blocks).
 *     Gradients have their input's shape and element type (d_xhat/d_bhat in xb_dtype;
 *     d_da, d_rot, d_initial fp32).
 *   - valid_len is a HOST array of b int64 values.  Positions t >= valid_len[b] contribute
 *     nothing and receive exactly zero gradient; values above s are clamped to s.
 *   - chunk_len must divide s.  It sets the granularity of the chunk-boundary carries; the
 *     result does not depend on it (the chunked recurrence is exact).
 *   - Every tensor pointer must be 16-byte aligned (as cudaMalloc and PyTorch allocations
 *     are); a misaligned one is rejected with MM_ERR_INVALID_ARG.
 *   - All device pointers are owned by the caller.  The library never allocates, frees or
 *     synchronises: every call only enqueues work on `stream` (a cudaStream_t; NULL = the
 *     legacy default stream) and returns.  Outputs are overwritten, never accumulated.
 *   - Stream capture: after a problem's first call on a device (which may set a kernel's
 *     shared-memory limit), calls of that problem issue nothing but stream work -- kernel
 *     launches and memsets -- so they can be recorded into a CUDA graph and replayed; the
 *     problem, its valid lengths and every pointer are fixed in the recorded graph.
 *   - `workspace` is caller-owned device scratch of at least mm_workspace_bytes() bytes,
 *     256-byte aligned.  Its contents need no initialisation and are clobbered.
 *   - Calls are thread-compatible: concurrent calls need distinct workspaces.
 *
 * Errors: arguments are validated on the host before anything is enqueued; a failed
 * validation returns an error and enqueues nothing.  MM_ERR_CUDA reports a launch error
 * (the stream may then hold partial work).  Device-side faults surface on the stream like
 * any CUDA error.
 */
#ifndef GB300_MOMENTS_H
#define GB300_MOMENTS_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MM_OK = 0,
    MM_ERR_INVALID_ARG = 1, /* shape/flag inconsistency, null pointer, chunk_len not dividing s ... */
    MM_ERR_UNSUPPORTED = 2, /* valid arguments outside what this build implements          */
    MM_ERR_WORKSPACE = 3,   /* workspace NULL, misaligned or smaller than mm_workspace_bytes */
    MM_ERR_CUDA = 4,        /* a CUDA launch or enqueue failed                              */
    MM_ERR_NONFINITE = 5,   /* MM_FLAG_CHECK_FINITE found a NaN / inf output (mm_device_status) */
    MM_ERR_TIMEOUT = 6      /* a bounded device-side wait gave up (mm_device_status)        */
} mm_status;

typedef enum { MM_F32 = 0, MM_BF16 = 1 } mm_dtype;

typedef enum {
    MM_ROT_NONE = 0,
    MM_ROT_PAIRWISE = 1, /* complex pairs (2i, 2i+1), i < rope_dim/2 ("rotate_chunk", interleaved) */
    MM_ROT_HALF = 2,     /* complex pairs (i, i + r/2), i < rope_dim/2 ("rotate_chunk", half-and-half) */
    MM_ROT_QUAT = 3      /* 4-blocks (4k..4k+3) = (w,x,y,z), k < quat_blocks ("rotate_chunk", quaternion) */
} mm_rot_kind;

/* Kernel-path selection (mm_problem.flags). */
#define MM_FLAG_FORCE_GENERIC 0x1u /* use the SIMT fp32 kernels even where the tensor-core path applies */
/* moments_bwd only: the workspace holds the chunk carries that a moments_fwd call with the same
 * problem and the same input tensors wrote into it (the caller sized that workspace with
 * mm_workspace_bytes(prob, 1) and passed it to both calls, and changed none of the inputs in
 * between).  The backward then skips recomputing the chunk-end contributions and the carry scan.
 * The flag is ignored (the carries are recomputed) when the forward and the backward of the
 * problem take different kernel paths (mm_path differs), whose carry layouts differ. */
#define MM_FLAG_REUSE_CARRIES 0x2u
/* Debug check of the results ("recalculated.rs", moments_phys_fwd: the `san` pass over (m2, m1)
 * after the chunk loop, read as a finiteness check that leaves the values unchanged): after its
 * kernels the call enqueues one more pass over its outputs (m2, m1; or the five gradients) that
 * marks the workspace if any element is NaN or infinite.  mm_device_status() then reports
 * MM_ERR_NONFINITE.  Off by default; it costs one read of the outputs. */
#define MM_FLAG_CHECK_FINITE 0x4u
/* The rotation is given as per-token steps instead of the cumulative rotation: `rot` holds angle
 * steps [b, s, h, rope_dim/2] (complex kinds) or quaternion steps [b, s, h, J, 4], and the library
 * builds the cumulative rotation the operator takes ("recalculated.rs", RotPrim: cumulative
 * angles / cumulative unit quaternions; their producer, RotationSeq / rotation::quat_mul, is named
 * there but not given).  Reading: angles theta_t = sum_{u<=t} dtheta_u (inclusive prefix sum along
 * the sequence); quaternions Q_t = q_t (x) Q_{t-1} from Q_{-1} = 1 (Hamilton product as
 * quat_mul_prim).  moments_bwd then returns in d_rot the gradient w.r.t. the steps (same shape as
 * `rot`): d_dtheta_u = sum_{t>=u} d_theta_t; G_t = dQ_t + conj(q_{t+1}) (x) G_{t+1},
 * d_q_t = G_t (x) conj(Q_{t-1}).  Steps past valid_len get zero gradient.  The build and its
 * gradient run as extra passes over [b, s, h, rw] in the workspace (mm_workspace_bytes counts
 * them when the flag is set); a backward that takes the forward's carries
 * (MM_FLAG_REUSE_CARRIES, honoured) also takes the cumulative rotation the forward built.
 * Ignored when the problem has no rotation. */
#define MM_FLAG_ROT_STEPS 0x8u
/* moments_fwd only, for testing the device failure path: on the tensor-core path every CTA of the
 * chunk-end kernel waits once, with a short poll limit, for an mbarrier phase that nothing
 * completes.  The bounded wait gives up, the kernels wind down without faulting or hanging, the
 * call's m2 / m1 are invalid, and mm_device_status() then reports MM_ERR_TIMEOUT; the next call
 * (without the flag) on the same stream and device runs normally.  Ignored on the SIMT path. */
#define MM_FLAG_TEST_WAIT_TIMEOUT 0x80000000u

typedef struct {
    int64_t b, s, C, h, p, r; /* batch, padded sequence, channels, heads, per-head dim, state rank */
    int64_t chunk_len;        /* l: divides s                                                     */
    int32_t xb_dtype;         /* mm_dtype of xhat / bhat and of their gradients                   */
    int32_t rot;              /* mm_rot_kind                                                      */
    int64_t rope_dim;         /* complex kinds: rotated width, even; pairwise <= r, half <= r     */
    int64_t quat_blocks;      /* quaternion kind: J, with 4*J <= r                                */
    uint32_t flags;           /* MM_FLAG_*                                                        */
    uint32_t reserved;
} mm_problem;

/* Bytes of device workspace a forward (backward = 0) or backward (backward != 0) call needs;
 * 0 if the problem is invalid.  Host-only, enqueues nothing. */
size_t mm_workspace_bytes(const mm_problem* prob, int backward);

/* Forward: (m2, m1) of the operator above.
 * Source: "recalculated.rs", Mamba3MomentsBackendExt::mamba3_state_moments_phys / moments_phys_fwd. */
mm_status moments_fwd(const mm_problem* prob, const void* xhat, const void* bhat, const float* da,
                      const float* rot, const float* initial, const int64_t* valid_len_host,
                      float* m2, float* m1, void* workspace, size_t ws_bytes, void* stream);

/* Backward: the five input gradients for cotangents (d_m2, d_m1), recomputing every state
 * from the leaf inputs (nothing is saved by the forward; with MM_FLAG_REUSE_CARRIES the chunk
 * carries, 1/chunk of the state trajectory, come from the forward's workspace instead).
 * d_m2 need not be symmetric.
 * Source: "backward.rs", moments_phys_bwd, MomentsGrads, module header "Gradient math". */
mm_status moments_bwd(const mm_problem* prob, const void* xhat, const void* bhat, const float* da,
                      const float* rot, const float* initial, const int64_t* valid_len_host,
                      const float* d_m2, const float* d_m1, void* d_xhat, void* d_bhat, float* d_da,
                      float* d_rot, float* d_initial, void* workspace, size_t ws_bytes, void* stream);

/* Static description of a status code (never NULL). */
const char* mm_status_string(mm_status status);

/* Which kernel path a call with this problem takes: 0 = SIMT fp32, 1 = tcgen05 tensor-core
 * path; -1 if the problem is invalid.  Host-only.  The tensor-core path takes bf16 operands with
 * p a multiple of 8 below 64 or of 64 up to 512, r a multiple of 16 up to 128 (64 or 128 for
 * half-split rotation),
 * any s, 1 <= C <= 8 and a rotation width (rope_dim / 2, or 4 quat_blocks) that is a multiple of 4
 * and at most 128. */
int mm_path(const mm_problem* prob, int backward);

/* ---- optional kernel timing (diagnostics; not needed to use the operator) ----
 * mm_profile_enable(1) clears previous records and makes every later call record a CUDA event
 * pair around each kernel it launches, on the call's stream (host overhead: a few microseconds
 * per launch).  mm_profile_enable(0) stops recording and keeps the records.
 * mm_profile_collect() waits for the recorded events and writes, per kernel id in [0, n), the
 * summed device milliseconds and the launch count; it returns the number of kernel ids (or -1
 * on a CUDA error).  mm_kernel_name() names a kernel id.  Process-global; not for concurrent use. */
void mm_profile_enable(int on);
int mm_profile_collect(double* total_ms, int64_t* launches, int n);
const char* mm_kernel_name(int id);

/* Reads the device status words a previous call left in `workspace` (synchronises `stream`).
 * MM_OK; MM_ERR_TIMEOUT if a bounded device-side wait of a tensor-core kernel gave up (the
 * outputs of that call are then invalid); MM_ERR_NONFINITE if the call ran with
 * MM_FLAG_CHECK_FINITE and an output holds a NaN or infinity; or MM_ERR_CUDA.
 * workspace == NULL reads the status of the last moments_fwd_noalloc call on the current device
 * (its fixed scratch holds the same words).  Diagnostic; calls never need it. */
mm_status mm_device_status(const void* workspace, void* stream);

/* ---- forward without a caller-provided workspace ----
 * The source pages have no counterpart to this call; it exists for callers that cannot
 * allocate device memory: code inside a host framework whose caching allocator owns every
 * device allocation, latency-critical loops where cudaMalloc / cudaFree may synchronise the
 * device, or plain C callers that hold only their input and output buffers.
 * It computes exactly what moments_fwd() computes, with the same arguments minus the workspace.
 * The scratch is a fixed 16 MiB array that the library keeps in device memory on every GPU that
 * loads it, until the process exits.  Problems whose forward workspace (mm_workspace_bytes(prob,
 * 0)) exceeds 16 MiB are rejected with MM_ERR_WORKSPACE before anything is enqueued.  The call
 * allocates nothing.  It runs on the current device; `stream` must belong to that device
 * (else MM_ERR_INVALID_ARG).  The first call on each device (and the first after that device's
 * context was reset) looks up the array's device address with that device current; make that
 * first call before any stream capture: made during a capture it returns MM_ERR_UNSUPPORTED.
 * Every call on a device shares the one array: calls that can overlap on the GPU (other
 * streams, other host threads) race on it, so the caller must serialise them.  The array keeps
 * the previous call's contents; each call initialises everything it reads.  Device-side status
 * (a bounded wait that gave up, MM_FLAG_CHECK_FINITE) is read with mm_device_status(NULL, stream). */
mm_status moments_fwd_noalloc(const mm_problem* prob, const void* xhat, const void* bhat, const float* da,
                              const float* rot, const float* initial, const int64_t* valid_len_host,
                              float* m2, float* m1, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* GB300_MOMENTS_H */
