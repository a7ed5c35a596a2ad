// debug_check.cuh -- bounds checks of computed global store indices.
//
// Compiled in only when MXFP8_DEBUG is defined (the library's debug build,
// libmxfp8_gb300_debug.so).  Every checked store tests its element range
// [idx, idx + len) against the extent of the buffer it writes, as derived
// from the call's shape; a store outside it is skipped and sets this
// translation unit's debug word, which mxfp8_device_error() reports as
// MXFP8_ERR_OUT_OF_BOUNDS.  Nothing traps.  In the normal build store_ok()
// is the constant true and the checks compile away.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace mxk {
namespace {

__device__ unsigned int g_oob_word;

#ifdef MXFP8_DEBUG
__device__ __forceinline__ bool store_ok(int64_t idx, int64_t len, int64_t extent) {
    if (idx >= 0 && len >= 0 && idx + len <= extent) return true;
    atomicOr(&g_oob_word, 1u);
    return false;
}
#else
__device__ __forceinline__ constexpr bool store_ok(int64_t, int64_t, int64_t) { return true; }
#endif

// Reads and clears this translation unit's debug word (always 0 in the
// normal build).
inline cudaError_t read_and_clear_oob_word(unsigned int* out) {
    unsigned int zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(out, g_oob_word, sizeof(unsigned int));
    if (e != cudaSuccess) return e;
    return cudaMemcpyToSymbol(g_oob_word, &zero, sizeof(unsigned int));
}

}  // namespace
}  // namespace mxk
