// dsa_internal.h -- helpers shared by the library's translation units
// (error messages for dsa_last_error(), device allocation with the test
// hook of dsa_debug_fail_alloc_after(), the projection behind
// dsa_decode_step_fused()).  Not part of the C ABI.
#pragma once

#include <cuda_runtime.h>

#include <cstddef>

struct dsa_proj_ctx;

namespace dsa_detail {

__attribute__((visibility("hidden"))) int fail(int code, const char *fmt, ...);
__attribute__((visibility("hidden"))) int cuda_fail(cudaError_t e, const char *what);
__attribute__((visibility("hidden"))) int dev_alloc(void **p, size_t bytes, const char *what);

// Records that `handle` (a decode or policy handle) launches a kernel on
// stream `st` next; true if the library's previous launch on `st` was for
// another handle (false for a stream not seen before).  forget_handle drops
// a destroyed handle from the record.
__attribute__((visibility("hidden"))) bool note_launch(cudaStream_t st, const void *handle);
__attribute__((visibility("hidden"))) void forget_handle(const void *handle);

// The QKV projection (dsa_proj.cu) as the fused decode step uses it.  k and
// v rows of stream s are written at k + s * kstride and v + s * vstride
// (elements; 0: head_dim, i.e. [batch * heads, head_dim] tensors), as bf16,
// or as E4M3 codes of fp32(value) * kinv[s] (vinv[s]) when those are given.
__attribute__((visibility("hidden"))) int proj_shape(const dsa_proj_ctx *p, int *batch, int *heads, int *head_dim);
__attribute__((visibility("hidden"))) void proj_staging(const dsa_proj_ctx *p, void **q);
__attribute__((visibility("hidden"))) int proj_launch(dsa_proj_ctx *p, const void *x, const void *W, int pos, void *q,
                                                      void *k, void *v, cudaStream_t st, int kstride = 0,
                                                      int vstride = 0, const float *kinv = nullptr,
                                                      const float *vinv = nullptr);

}  // namespace dsa_detail
