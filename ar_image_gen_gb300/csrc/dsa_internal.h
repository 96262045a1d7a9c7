// dsa_internal.h -- helpers shared by the library's translation units
// (error messages for dsa_last_error(), device allocation with the test
// hook of dsa_debug_fail_alloc_after()).  Not part of the C ABI.
#pragma once

#include <cuda_runtime.h>

#include <cstddef>

namespace dsa_detail {

__attribute__((visibility("hidden"))) int fail(int code, const char *fmt, ...);
__attribute__((visibility("hidden"))) int cuda_fail(cudaError_t e, const char *what);
__attribute__((visibility("hidden"))) int dev_alloc(void **p, size_t bytes, const char *what);

}  // namespace dsa_detail
