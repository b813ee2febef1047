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

// Unique id of the current CUDA context (0 if none is current or the driver
// cannot say). Set-up that belongs to a context (kernel attributes, device
// addresses of the library's own arrays) is cached under this id and redone
// when it changes, e.g. after cudaDeviceReset destroyed the old context.
unsigned long long context_id();

cudaError_t launch_prefill_f32(const float *q, const float *k, const float *v, const float *r,
                               float *out, float *lse, int B, int Hq, int Hkv, int L, int d,
                               unsigned *err, cudaStream_t stream);

// Returns cudaErrorInvalidValue if a tensor map could not be encoded.
// 3-D bf16 tensor map over [heads][L][128] with 128-byte swizzle and boxes
// of box_rows x 64 elements (zero fill past L).
bool make_head_rows_map(EncodeTiledFn enc, CUtensorMap *map, const void *ptr, int L, int heads,
                        int box_rows);

// L queries, the last L positions of Lk >= L keys (Lk == L: plain prefill).
// lse, cor (|correction| / |o| per row), o1 (bf16 o^SA per row) and sbar
// (sigma / l per row) may each be null.
cudaError_t launch_prefill_tc(const void *q, const void *k, const void *v, const void *r, void *out,
                              float *lse, float *cor, void *o1, float *sbar, int B, int Hq, int Hkv,
                              int L, int Lk, unsigned *err, cudaStream_t stream);

// Backward of the causal prefill (Lq == Lk == L, d = 128, bf16). stats is a
// workspace of B * Hq * round_up(L, 64) float4 records.
size_t prefill_bwd_stats_count(int B, int Hq, int L);
cudaError_t launch_prefill_bwd(const void *q, const void *k, const void *v, const void *r,
                               const void *out, const void *o1, const float *lse,
                               const float *sbar, const void *dout, void *dq, void *dk, void *dv,
                               void *dr, int B, int Hq, int Hkv, int L, void *stats, unsigned *err,
                               cudaStream_t stream);

// Decode over nshare CTAs, each with an equal share of the batch's keys (all
// sequences and kv heads in one stream). default_share: the default
// schedule, which also gives every CTA at least 512 keys (fewer CTAs take
// part in small batches); otherwise min(nshare, keys) CTAs take part.
// cor ([B, Hq] fp32, |correction| / |o|) may be null.
cudaError_t launch_decode(const void *q, const void *r, const void *kcache, const void *vcache,
                          const int *seqlens, void *out, float *cor, int B, int Hq, int Hkv,
                          int nshare, bool default_share, void *workspace, unsigned *err,
                          cudaStream_t stream);

// Decode workspace: a table of {first record slot, slots} per (sequence, kv
// head), padded to 256 bytes, then (nshare + B * Hkv) slots of Hq / Hkv
// records of 2 d + 2 floats. CTA c writes its part of row `row` (sequence,
// kv head) to slot c + row; a later CTA never holds an earlier row, so the
// slots of the (CTA, row) pairs that meet are distinct.
inline size_t decode_meta_bytes(int B, int Hkv) {
  return (static_cast<size_t>(B) * Hkv * 8 + 255) / 256 * 256;
}
inline size_t decode_workspace_bytes(int B, int Hq, int Hkv, int d, int nshare) {
  const size_t recs = static_cast<size_t>(nshare) * (Hq / Hkv) + static_cast<size_t>(B) * Hq;
  return decode_meta_bytes(B, Hkv) + recs * (2 * static_cast<size_t>(d) + 2) * sizeof(float);
}

// Fixed split-record array of the allocation-free decode: 16 MiB of fp32.
constexpr size_t kNoAllocScratchFloats = size_t(4) << 20;
// Device address of that array on the current device (resolved once per device).
cudaError_t noalloc_scratch(float **ptr);

// Fused [W_Q; W_K; W_V; W_R] x projection into per-head q, k, v, r (d = 128).
cudaError_t launch_qkvr_proj(const void *x, const void *w, void *q, void *k, void *v, void *r,
                             int B, int L, int D, int Hq, int Hkv, unsigned *err,
                             cudaStream_t stream);

cudaError_t launch_timeout_probe(long long limit_cycles, unsigned *err, cudaStream_t stream);

}  // namespace plx
