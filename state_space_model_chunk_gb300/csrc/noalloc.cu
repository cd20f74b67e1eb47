// noalloc.cu -- moments_fwd_noalloc: the forward for callers that cannot allocate device memory.
//
// Some callers cannot hand the library a workspace: code embedded in a host framework whose
// caching allocator owns every device allocation, latency-critical loops where cudaMalloc or
// cudaFree may synchronise the device, or plain C callers that hold nothing but their input and
// output buffers.  This entry point runs the ordinary forward with its scratch placed in a
// fixed array that lives in device memory for as long as the library is loaded.
#include <mutex>

#include "../../include/moments.h"
#include <cuda_runtime.h>

namespace {

// 16 MiB of scratch on every GPU that loads the library, held until the process exits.
constexpr size_t kNoAllocScratchBytes = (size_t)16 << 20;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
void* g_noalloc_ptr[kMaxDevices];  // device address of g_noalloc_scratch, looked up once per device

}  // namespace

extern "C" mm_status moments_fwd_noalloc(const mm_problem* prob, const void* xhat, const void* bhat,
                                         const float* da, const float* rot, const float* initial,
                                         const int64_t* valid_len_host, float* m2, float* m1, void* stream) {
    const size_t need = mm_workspace_bytes(prob, 0);
    if (need == 0) return MM_ERR_INVALID_ARG;
    if (need > kNoAllocScratchBytes) return MM_ERR_WORKSPACE;  // problem too large for the fixed scratch
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return MM_ERR_CUDA;
    }
    if (dev < 0 || dev >= kMaxDevices) return MM_ERR_UNSUPPORTED;
    void* scratch = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_noalloc_mu);
        if (!g_noalloc_ptr[dev]) {
            // The host-side name of the array is only a stand-in; the kernel needs the device address.
            void* p = nullptr;
            if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
                cudaGetLastError();
                return MM_ERR_CUDA;
            }
            g_noalloc_ptr[dev] = p;
        }
        scratch = g_noalloc_ptr[dev];
    }
    // The forward initialises everything it reads in its workspace (error word, carries), so
    // the contents left by an earlier call do not matter.
    return moments_fwd(prob, xhat, bhat, da, rot, initial, valid_len_host, m2, m1, scratch,
                       kNoAllocScratchBytes, stream);
}
