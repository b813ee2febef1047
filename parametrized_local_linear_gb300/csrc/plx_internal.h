// Host-side interface between the C ABI (capi.cu) and the kernel translation
// units. Arguments arrive here already validated.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>

namespace plx {

// Device error word of the current device (bit kErrTimeout = a bounded wait
// ran out). Null if it could not be resolved.
unsigned *device_error_word();

// cuTensorMapEncodeTiled resolved through the runtime (no libcuda link).
using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn encode_tiled_fn();

int sm_count();

cudaError_t launch_prefill_f32(const float *q, const float *k, const float *v, const float *r,
                               float *out, float *lse, int B, int Hq, int Hkv, int L, int d,
                               unsigned *err, cudaStream_t stream);

// Returns cudaErrorInvalidValue if a tensor map could not be encoded.
// L queries, the last L positions of Lk >= L keys (Lk == L: plain prefill).
// lse and cor (|correction| / |o| per row) may be null.
cudaError_t launch_prefill_tc(const void *q, const void *k, const void *v, const void *r, void *out,
                              float *lse, float *cor, int B, int Hq, int Hkv, int L, int Lk,
                              unsigned *err, cudaStream_t stream);

// cor ([B, Hq] fp32, |correction| / |o|) may be null.
cudaError_t launch_decode(const void *q, const void *r, const void *kcache, const void *vcache,
                          const int *seqlens, void *out, float *cor, int B, int Hq, int Hkv,
                          int nsplit, float *workspace, unsigned *err, cudaStream_t stream);

// Fixed split-record array of the allocation-free decode: 16 MiB of fp32.
constexpr size_t kNoAllocScratchFloats = size_t(4) << 20;
// Device address of that array on the current device (resolved once per device).
cudaError_t noalloc_scratch(float **ptr);

cudaError_t launch_timeout_probe(long long limit_cycles, unsigned *err, cudaStream_t stream);

}  // namespace plx
