// noalloc.h -- the fixed device scratch behind moments_fwd_noalloc (noalloc.cu), for abi.cu.
#pragma once
#include <stddef.h>

#include "../../include/moments.h"

// Bytes of the fixed scratch array.
size_t noalloc_scratch_bytes();
// Device address of the fixed scratch array on the current device (looked up on first use in
// the current context; MM_ERR_UNSUPPORTED if that first look-up would happen while `stream` is
// being captured).
mm_status noalloc_scratch(void* stream, void** out);
