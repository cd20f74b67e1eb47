// fast_bwd_rag.cu -- the backward kernel's general-shape instantiations, for sequence lengths that
// are not a multiple of 64 and for fewer than 64 state rows per head (compiled apart from
// fast_bwd.cu so that the two build in parallel).
#include "fast_bwd_kernel.cuh"

namespace fastbwd {

BwdKernel ragged_bwd_kernel(int rot, int layoutB, bool c8) {
#define BWD_KERN(K, L) (c8 ? tc_bwd_kernel<K, L, 3, true> : tc_bwd_kernel<K, L, 2, true>)
    switch (rot) {
        case ROT_PAIRWISE: return BWD_KERN(ROT_PAIRWISE, 0);
        case ROT_HALF: return layoutB ? BWD_KERN(ROT_HALF, 1) : BWD_KERN(ROT_HALF, 0);
        case ROT_QUAT: return BWD_KERN(ROT_QUAT, 0);
        default: return BWD_KERN(ROT_NONE, 0);
    }
#undef BWD_KERN
}

}  // namespace fastbwd
