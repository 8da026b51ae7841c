// Device-side error word.  Kernels record the first failure they see (a
// bounded wait that ran out, or a failed in-kernel check) here and return;
// the host reads and clears it with w8a8_get_device_error().  The word has
// internal linkage, so each translation unit that includes this header owns
// its own copy and exposes it through its own host accessor.
#pragma once
#include <cstdint>

#define W8A8_DEVERR_NONE 0
// 0x100 + site: a bounded mbarrier wait ran out at the numbered site.
#define W8A8_DEVERR_TIMEOUT_BASE 0x100

namespace w8a8 {

static __device__ unsigned int g_device_error;

__device__ __forceinline__ void record_device_error(unsigned int code) {
    atomicCAS(&g_device_error, 0u, code);
}

__device__ __forceinline__ bool device_error_set() {
    return *(volatile unsigned int*)&g_device_error != 0u;
}

}  // namespace w8a8
