// noalloc.cu -- moments_fwd_noalloc: the forward for callers that cannot allocate device memory.
//
// Some callers cannot hand the library a workspace: code embedded in a host framework whose
// caching allocator owns every device allocation, latency-critical loops where cudaMalloc or
// cudaFree may synchronise the device, or plain C callers that hold nothing but their input and
// output buffers.  This entry point runs the ordinary forward with its scratch placed in a
// fixed array that lives in device memory for as long as the library is loaded.
#include <cuda.h>

#include <mutex>

#include "../../include/moments.h"
#include <cuda_runtime.h>

#include "noalloc.h"

namespace {

// 16 MiB of scratch on every GPU that loads the library, held until the process exits.
constexpr size_t kNoAllocScratchBytes = (size_t)16 << 20;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
// Device address of g_noalloc_scratch per device, and the context it was looked up in: a
// context torn down and created again (cudaDeviceReset) places the module anew, so the address
// is looked up again whenever the device's current context is not the one it was found in.
void* g_noalloc_ptr[kMaxDevices];
CUcontext g_noalloc_ctx[kMaxDevices];

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);

CtxGetCurrentFn ctx_get_current() {
    static CtxGetCurrentFn fn = nullptr;
    static bool tried = false;
    if (!tried) {
        tried = true;
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<CtxGetCurrentFn>(p);
        else
            cudaGetLastError();
    }
    return fn;
}

}  // namespace

size_t noalloc_scratch_bytes() { return kNoAllocScratchBytes; }

mm_status noalloc_scratch(void* stream, void** out) {
    *out = nullptr;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return MM_ERR_CUDA;
    }
    if (dev < 0 || dev >= kMaxDevices) return MM_ERR_UNSUPPORTED;
    // the scratch and the kernels are those of the current device: a stream of another device
    // would run them against memory it does not own
    int sdev = dev;
    if (cudaStreamGetDevice(static_cast<cudaStream_t>(stream), &sdev) != cudaSuccess) {
        cudaGetLastError();
        return MM_ERR_CUDA;
    }
    if (sdev != dev) return MM_ERR_INVALID_ARG;
    CUcontext ctx = nullptr;
    CtxGetCurrentFn get = ctx_get_current();
    if (!get || get(&ctx) != CUDA_SUCCESS) return MM_ERR_CUDA;
    if (!ctx) {  // no context bound to this host thread yet: bind the device's primary context
        if (cudaSetDevice(dev) != cudaSuccess || get(&ctx) != CUDA_SUCCESS || !ctx) {
            cudaGetLastError();
            return MM_ERR_CUDA;
        }
    }
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (!g_noalloc_ptr[dev] || g_noalloc_ctx[dev] != ctx) {
        // The look-up may load the module; inside a stream capture that is not allowed, so the
        // first call on a device (or after a context reset) must come before any capture.
        cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
        if (cudaStreamIsCapturing(static_cast<cudaStream_t>(stream), &cap) != cudaSuccess) {
            cudaGetLastError();
            return MM_ERR_CUDA;
        }
        if (cap != cudaStreamCaptureStatusNone) return MM_ERR_UNSUPPORTED;
        // The host-side name of the array is only a stand-in; the kernels need the device address.
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
            cudaGetLastError();
            return MM_ERR_CUDA;
        }
        g_noalloc_ptr[dev] = p;
        g_noalloc_ctx[dev] = ctx;
    }
    *out = g_noalloc_ptr[dev];
    return MM_OK;
}

extern "C" mm_status moments_fwd_noalloc(const mm_problem* prob, const void* xhat, const void* bhat,
                                         const float* da, const float* rot, const float* initial,
                                         const int64_t* valid_len_host, float* m2, float* m1, void* stream) {
    const size_t need = mm_workspace_bytes(prob, 0);
    if (need == 0) return MM_ERR_INVALID_ARG;
    if (need > kNoAllocScratchBytes) return MM_ERR_WORKSPACE;  // problem too large for the fixed scratch
    void* scratch = nullptr;
    const mm_status st = noalloc_scratch(stream, &scratch);
    if (st != MM_OK) return st;
    // The forward initialises everything it reads in its workspace (status words, carries), so
    // the contents left by an earlier call do not matter.
    return moments_fwd(prob, xhat, bhat, da, rot, initial, valid_len_host, m2, m1, scratch,
                       kNoAllocScratchBytes, stream);
}
