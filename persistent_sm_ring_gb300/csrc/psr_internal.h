// Declarations shared between the library's translation units.  Not part of the C ABI: the
// library is built with hidden visibility, and only the functions of include/psr.h are exported.
#pragma once
#include <stddef.h>

#include "../../include/psr.h"

extern "C" {
// Checks the arguments of a forward call the way psr_ring_attn_fwd does, short of the
// workspace, and in the same order: null or misaligned q, k, v, o, lse -> PSR_ERR_ARG; no usable
// sm_103 device -> PSR_ERR_CUDA or PSR_ERR_UNSUPPORTED; the shape -> PSR_ERR_ARG or
// PSR_ERR_UNSUPPORTED.  On PSR_OK, *ws_need (if not NULL) is the workspace the shape needs on
// the current device.
int psr_internal_fwd_check(const psr_shape* shape, const void* q, const void* k, const void* v, const void* o,
                           const void* lse, size_t* ws_need);
}
