// prof.h -- optional CUDA-event timing of every kernel launch (off unless mm_profile_enable(1)).
#pragma once
#include <cuda_runtime.h>

enum MMKernelId {
    KID_CHUNK_END = 0,
    KID_CARRY_SCAN,
    KID_FWD_CHUNK,
    KID_DSYM,
    KID_BWD_CHUNK,
    KID_COT_SCAN,
    KID_CORRECT,
    KID_FAST_FWD,
    KID_FAST_END,
    KID_FAST_BWD,
    KID_FAST_CORRECT,
    KID_FINITE,
    KID_M2_REDUCE,
    KID_DROT_SUM,
    KID_ROT_STEPS,
    KID_GROUP_SUM,
    KID_COUNT
};

// Records an event on `st` before (begin = 1) or after (begin = 0) launch `kid` when profiling is on.
void mm_prof_mark(int kid, int begin, cudaStream_t st);

// cudaFuncSetAttribute(fn, MaxDynamicSharedMemorySize, bytes) on the current device, skipped when
// an earlier call already allowed at least `bytes` there: after a first call of a problem, the
// library's calls issue nothing but stream work (so a stream capture of them records only that).
cudaError_t mm_allow_smem(const void* fn, int bytes);
