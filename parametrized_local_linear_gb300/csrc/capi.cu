// C ABI of libplx.so: argument validation, per-device set-up, the decode
// workspace, device error reporting. The operations themselves are defined
// in include/plx.h; the kernels live in prefill_tc.cu, prefill_f32.cu and
// decode.cu.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdarg.h>
#include <stdio.h>

#include <algorithm>
#include <mutex>

#include "../../include/plx.h"
#include "plx_device.cuh"
#include "plx_internal.h"

namespace {

thread_local char g_msg[512] = "";

plx_status fail(plx_status s, const char *fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
  va_end(ap);
  return s;
}

plx_status cuda_fail(cudaError_t e, const char *what) {
  return fail(PLX_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Device error word: one per device (a __device__ variable is instantiated per
// device), its address resolved once per device.
__device__ unsigned g_plx_device_error = 0;

constexpr int kMaxDevices = 64;
std::mutex g_mu;
// Address of the error word per device, with the id of the context it was
// resolved in: a device reset destroys that context, and the next call
// resolves the address again in the new one.
unsigned *g_err_ptr[kMaxDevices] = {};
unsigned long long g_err_ctx[kMaxDevices] = {};
int g_sm_count[kMaxDevices] = {};

using CtxGetCurrentFn = CUresult (*)(CUcontext *);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long *);

int current_device() {
  int dev = 0;
  cudaGetDevice(&dev);
  return dev;
}

// Probe kernel for the bounded-wait failure path: wait on an mbarrier that
// nothing will ever arrive on.
__global__ void timeout_probe_kernel(long long limit, unsigned *err) {
  __shared__ uint64_t bar;
  __shared__ int flag;
  if (threadIdx.x == 0) {
    plx::mbar_init(plx::smem_u32(&bar), 1);
    flag = 0;
    plx::fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const plx::Abort ab{&flag, err};
    plx::mbar_wait(plx::smem_u32(&bar), 0, ab, limit);
  }
}

}  // namespace

namespace plx {

unsigned long long context_id() {
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<CtxGetCurrentFn>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<CtxGetIdFn>(p);
  });
  if (get_current == nullptr || get_id == nullptr) return 0;
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr || get_id(ctx, &id) != CUDA_SUCCESS)
    return 0;
  return id;
}

unsigned *device_error_word() {
  const int dev = current_device();
  if (dev < 0 || dev >= kMaxDevices) return nullptr;
  const unsigned long long ctx = context_id();
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_err_ptr[dev] == nullptr || ctx == 0 || g_err_ctx[dev] != ctx) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_plx_device_error) != cudaSuccess) return nullptr;
    g_err_ptr[dev] = static_cast<unsigned *>(p);
    g_err_ctx[dev] = ctx;
  }
  return g_err_ptr[dev];
}

int sm_count() {
  const int dev = current_device();
  if (dev < 0 || dev >= kMaxDevices) return 148;
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_sm_count[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 148;
    g_sm_count[dev] = n;
  }
  return g_sm_count[dev];
}

EncodeTiledFn encode_tiled_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

cudaError_t launch_timeout_probe(long long limit_cycles, unsigned *err, cudaStream_t stream) {
  timeout_probe_kernel<<<1, 32, 0, stream>>>(limit_cycles, err);
  return cudaGetLastError();
}

}  // namespace plx

namespace {

plx_status check_common(const char *fn, int B, int Hq, int Hkv, int L, int d) {
  if (B < 1 || Hq < 1 || Hkv < 1 || L < 1 || d < 1)
    return fail(PLX_ERR_INVALID_ARG, "%s: sizes must be >= 1 (B=%d Hq=%d Hkv=%d L=%d d=%d)", fn, B,
                Hq, Hkv, L, d);
  if (Hq % Hkv != 0)
    return fail(PLX_ERR_INVALID_ARG, "%s: Hq (%d) must be a multiple of Hkv (%d)", fn, Hq, Hkv);
  return PLX_OK;
}

plx_status finish_launch(cudaError_t e, const char *fn) {
  if (e != cudaSuccess) return cuda_fail(e, fn);
  return PLX_OK;
}

}  // namespace

extern "C" {

namespace {

plx_status prefill_bf16(const char *fn, const void *q, const void *k, const void *v, const void *r,
                        void *out, float *lse, float *cor, void *o1, float *sbar, int B, int Hq,
                        int Hkv, int Lq, int Lk, int d, void *stream) {
  if (!q || !k || !v || !r || !out) return fail(PLX_ERR_INVALID_ARG, "%s: null tensor pointer", fn);
  plx_status s = check_common(fn, B, Hq, Hkv, Lq, d);
  if (s) return s;
  if (Lk < Lq) return fail(PLX_ERR_INVALID_ARG, "%s: Lk (%d) must be >= Lq (%d)", fn, Lk, Lq);
  if (d != 128) return fail(PLX_ERR_UNSUPPORTED, "%s: head dim %d (only 128)", fn, d);
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(r) || !aligned16(out) ||
      !aligned16(o1))
    return fail(PLX_ERR_INVALID_ARG, "%s: tensor pointers must be 16-byte aligned", fn);
  if (static_cast<long long>(Lq + 127) / 128 * Hq * B > 0x7fffffffLL ||
      static_cast<long long>(B) * Hq > 0x7fffffff)
    return fail(PLX_ERR_UNSUPPORTED, "%s: problem too large for one launch", fn);
  return finish_launch(plx::launch_prefill_tc(q, k, v, r, out, lse, cor, o1, sbar, B, Hq, Hkv, Lq, Lk,
                                              plx::device_error_word(),
                                              static_cast<cudaStream_t>(stream)),
                       fn);
}

}  // namespace

plx_status plx_prefill_fwd_chunk(const void *q, const void *k, const void *v, const void *r,
                                 void *out, float *lse, int B, int Hq, int Hkv, int Lq, int Lk,
                                 int d, void *stream) {
  return prefill_bf16("plx_prefill_fwd", q, k, v, r, out, lse, nullptr, nullptr, nullptr, B, Hq, Hkv,
                      Lq, Lk, d, stream);
}

plx_status plx_prefill_fwd_cor(const void *q, const void *k, const void *v, const void *r,
                               void *out, float *lse, float *cor, int B, int Hq, int Hkv, int Lq,
                               int Lk, int d, void *stream) {
  if (!cor) return fail(PLX_ERR_INVALID_ARG, "plx_prefill_fwd_cor: null cor pointer");
  return prefill_bf16("plx_prefill_fwd_cor", q, k, v, r, out, lse, cor, nullptr, nullptr, B, Hq, Hkv,
                      Lq, Lk, d, stream);
}

plx_status plx_prefill_fwd_train(const void *q, const void *k, const void *v, const void *r,
                                 void *out, float *lse, void *o1, float *sbar, int B, int Hq,
                                 int Hkv, int L, int d, void *stream) {
  const char *fn = "plx_prefill_fwd_train";
  if (!lse || !o1 || !sbar) return fail(PLX_ERR_INVALID_ARG, "%s: null lse, o1 or sbar", fn);
  return prefill_bf16(fn, q, k, v, r, out, lse, nullptr, o1, sbar, B, Hq, Hkv, L, L, d, stream);
}

plx_status plx_prefill_bwd(const void *q, const void *k, const void *v, const void *r,
                           const void *out, const void *o1, const float *lse, const float *sbar,
                           const void *dout, void *dq, void *dk, void *dv, void *dr, int B, int Hq,
                           int Hkv, int L, int d, void *stream) {
  const char *fn = "plx_prefill_bwd";
  if (!q || !k || !v || !r || !out || !o1 || !lse || !sbar || !dout || !dq || !dk || !dv || !dr)
    return fail(PLX_ERR_INVALID_ARG, "%s: null pointer", fn);
  plx_status s = check_common(fn, B, Hq, Hkv, L, d);
  if (s) return s;
  if (d != 128) return fail(PLX_ERR_UNSUPPORTED, "%s: head dim %d (only 128)", fn, d);
  const void *ptrs[] = {q, k, v, r, out, o1, dout, dq, dk, dv, dr};
  for (const void *p : ptrs)
    if (!aligned16(p)) return fail(PLX_ERR_INVALID_ARG, "%s: tensor pointers must be 16-byte aligned", fn);
  if (static_cast<long long>(L + 127) / 128 * Hq * B > 0x7fffffffLL)
    return fail(PLX_ERR_UNSUPPORTED, "%s: problem too large for one launch", fn);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  void *ws = nullptr;
  const size_t need = plx::prefill_bwd_stats_count(B, Hq, L) * 4 * sizeof(float);
  cudaError_t e = cudaMallocAsync(&ws, need, st);
  if (e != cudaSuccess) return cuda_fail(e, "plx_prefill_bwd: workspace allocation");
  e = plx::launch_prefill_bwd(q, k, v, r, out, o1, lse, sbar, dout, dq, dk, dv, dr, B, Hq, Hkv, L,
                              ws, plx::device_error_word(), st);
  cudaError_t e2 = cudaFreeAsync(ws, st);
  if (e != cudaSuccess) return cuda_fail(e, fn);
  if (e2 != cudaSuccess) return cuda_fail(e2, "plx_prefill_bwd: workspace release");
  return PLX_OK;
}

plx_status plx_prefill_fwd(const void *q, const void *k, const void *v, const void *r, void *out,
                           float *lse, int B, int Hq, int Hkv, int L, int d, void *stream) {
  return plx_prefill_fwd_chunk(q, k, v, r, out, lse, B, Hq, Hkv, L, L, d, stream);
}

plx_status plx_prefill_fwd_f32(const float *q, const float *k, const float *v, const float *r,
                               float *out, float *lse, int B, int Hq, int Hkv, int L, int d,
                               void *stream) {
  const char *fn = "plx_prefill_fwd_f32";
  if (!q || !k || !v || !r || !out) return fail(PLX_ERR_INVALID_ARG, "%s: null tensor pointer", fn);
  plx_status s = check_common(fn, B, Hq, Hkv, L, d);
  if (s) return s;
  if (d != 64 && d != 128) return fail(PLX_ERR_UNSUPPORTED, "%s: head dim %d (64 or 128)", fn, d);
  if (B > 65535 || Hq > 65535)
    return fail(PLX_ERR_UNSUPPORTED, "%s: B and Hq must be <= 65535", fn);
  return finish_launch(plx::launch_prefill_f32(q, k, v, r, out, lse, B, Hq, Hkv, L, d,
                                               plx::device_error_word(),
                                               static_cast<cudaStream_t>(stream)),
                       fn);
}

plx_status plx_qkvr_proj(const void *x, const void *w, void *q, void *k, void *v, void *r, int B,
                         int L, int D, int Hq, int Hkv, int d, void *stream) {
  const char *fn = "plx_qkvr_proj";
  if (!x || !w || !q || !k || !v || !r) return fail(PLX_ERR_INVALID_ARG, "%s: null pointer", fn);
  plx_status s = check_common(fn, B, Hq, Hkv, L, d);
  if (s) return s;
  if (D < 1 || D % 8 != 0)
    return fail(PLX_ERR_INVALID_ARG, "%s: model dim %d must be a positive multiple of 8", fn, D);
  if (d != 128) return fail(PLX_ERR_UNSUPPORTED, "%s: head dim %d (only 128)", fn, d);
  const void *ptrs[] = {x, w, q, k, v, r};
  for (const void *p : ptrs)
    if (!aligned16(p)) return fail(PLX_ERR_INVALID_ARG, "%s: pointers must be 16-byte aligned", fn);
  if (static_cast<long long>(B) * L > 0x7fffffffLL - 128 ||
      static_cast<long long>(2 * Hq + 2 * Hkv) * d > 0x7fffffffLL)
    return fail(PLX_ERR_UNSUPPORTED, "%s: problem too large for one launch", fn);
  return finish_launch(plx::launch_qkvr_proj(x, w, q, k, v, r, B, L, D, Hq, Hkv,
                                             plx::device_error_word(),
                                             static_cast<cudaStream_t>(stream)),
                       fn);
}

size_t plx_decode_workspace_bytes(int B, int Hq, int Hkv, int d, int nsplit) {
  if (B < 1 || Hq < 1 || Hkv < 1 || d < 1 || nsplit < 1 || Hq % Hkv != 0) return 0;
  return plx::decode_workspace_bytes(B, Hq, Hkv, d, nsplit);
}

int plx_decode_default_nsplit(int B, int Hkv) {
  (void)B;
  (void)Hkv;
  // One wave of the split kernel: two CTAs fit on an SM (its registers), and
  // every CTA takes an equal share of the batch's keys, so a single wave keeps
  // every SM streaming until the end with no tail. Lengths live on the
  // device, so the kernel itself lowers the count for small batches
  // (floor(sqrt(W)) CTAs for W keys). Measured on GB300 with per-sequence splits before this
  // schedule: uniform batches ran fastest at 256 CTAs (B = 1..32, 8192
  // tokens), a ragged one (B = 8, 16k-131k tokens) needed 32 splits a
  // sequence to even out its lengths.
  return 2 * plx::sm_count();
}

namespace {

plx_status check_decode_args(const char *fn, const void *q, const void *r, const void *kcache,
                             const void *vcache, const int *seqlens, void *out, int B, int Hq,
                             int Hkv, int d) {
  if (!q || !r || !kcache || !vcache || !seqlens || !out)
    return fail(PLX_ERR_INVALID_ARG, "%s: null pointer", fn);
  plx_status s = check_common(fn, B, Hq, Hkv, 1, d);
  if (s) return s;
  if (d != 128) return fail(PLX_ERR_UNSUPPORTED, "%s: head dim %d (only 128)", fn, d);
  if (Hq / Hkv > 8) return fail(PLX_ERR_UNSUPPORTED, "%s: Hq / Hkv = %d (at most 8)", fn, Hq / Hkv);
  if (static_cast<long long>(B) * Hq > (1LL << 24))
    return fail(PLX_ERR_UNSUPPORTED, "%s: B * Hq must be <= 2^24", fn);
  if (!aligned16(q) || !aligned16(r) || !aligned16(kcache) || !aligned16(vcache) || !aligned16(out))
    return fail(PLX_ERR_INVALID_ARG, "%s: tensor pointers must be 16-byte aligned", fn);
  return PLX_OK;
}

plx_status decode_bf16(const char *fn, const void *q, const void *r, const void *kcache,
                       const void *vcache, const int *seqlens, void *out, float *cor, int B,
                       int Hq, int Hkv, int d, int nsplit, bool default_share, void *workspace,
                       size_t workspace_bytes, void *stream) {
  plx_status s = check_decode_args(fn, q, r, kcache, vcache, seqlens, out, B, Hq, Hkv, d);
  if (s) return s;
  if (nsplit < 1) return fail(PLX_ERR_INVALID_ARG, "%s: nsplit %d", fn, nsplit);
  if (nsplit > 65535) return fail(PLX_ERR_INVALID_ARG, "%s: nsplit %d too large", fn, nsplit);
  const size_t need = plx::decode_workspace_bytes(B, Hq, Hkv, d, nsplit);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (workspace != nullptr) {
    if (workspace_bytes < need)
      return fail(PLX_ERR_INVALID_ARG, "%s: workspace of %zu bytes, need %zu", fn, workspace_bytes,
                  need);
    if (!aligned16(workspace)) return fail(PLX_ERR_INVALID_ARG, "%s: workspace not 16-byte aligned", fn);
    return finish_launch(plx::launch_decode(q, r, kcache, vcache, seqlens, out, cor, B, Hq, Hkv,
                                            nsplit, default_share, workspace,
                                            plx::device_error_word(), st),
                         fn);
  }
  void *ws = nullptr;
  cudaError_t e = cudaMallocAsync(&ws, need, st);
  if (e != cudaSuccess) return cuda_fail(e, "plx_decode_fwd: workspace allocation");
  e = plx::launch_decode(q, r, kcache, vcache, seqlens, out, cor, B, Hq, Hkv, nsplit,
                         default_share, ws, plx::device_error_word(), st);
  cudaError_t e2 = cudaFreeAsync(ws, st);
  if (e != cudaSuccess) return cuda_fail(e, fn);
  if (e2 != cudaSuccess) return cuda_fail(e2, "plx_decode_fwd: workspace release");
  return PLX_OK;
}

}  // namespace

plx_status plx_decode_fwd_ex(const void *q, const void *r, const void *kcache, const void *vcache,
                             const int *seqlens, void *out, int B, int Hq, int Hkv, int d,
                             int nsplit, void *workspace, size_t workspace_bytes, void *stream) {
  const bool default_share = nsplit <= 0;
  return decode_bf16("plx_decode_fwd", q, r, kcache, vcache, seqlens, out, nullptr, B, Hq, Hkv, d,
                     default_share ? plx_decode_default_nsplit(B, Hkv) : nsplit, default_share,
                     workspace, workspace_bytes, stream);
}

plx_status plx_decode_fwd_cor(const void *q, const void *r, const void *kcache, const void *vcache,
                              const int *seqlens, void *out, float *cor, int B, int Hq, int Hkv,
                              int d, void *stream) {
  if (!cor) return fail(PLX_ERR_INVALID_ARG, "plx_decode_fwd_cor: null cor pointer");
  return decode_bf16("plx_decode_fwd_cor", q, r, kcache, vcache, seqlens, out, cor, B, Hq, Hkv, d,
                     plx_decode_default_nsplit(B, Hkv), true, nullptr, 0, stream);
}

plx_status plx_decode_fwd(const void *q, const void *r, const void *kcache, const void *vcache,
                          const int *seqlens, void *out, int B, int Hq, int Hkv, int d,
                          void *stream) {
  return plx_decode_fwd_ex(q, r, kcache, vcache, seqlens, out, B, Hq, Hkv, d, 0, nullptr, 0,
                           stream);
}

plx_status plx_decode_fwd_noalloc(const void *q, const void *r, const void *kcache,
                                  const void *vcache, const int *seqlens, void *out, int B, int Hq,
                                  int Hkv, int d, void *stream) {
  const char *fn = "plx_decode_fwd_noalloc";
  const size_t cap_bytes = plx::kNoAllocScratchFloats * sizeof(float);
  // Arguments are checked before the array's address is looked up, so a
  // rejected call makes no CUDA call at all.
  plx_status s = check_decode_args(fn, q, r, kcache, vcache, seqlens, out, B, Hq, Hkv, d);
  if (s) return s;
  const size_t one = plx_decode_workspace_bytes(B, Hq, Hkv, d, 1);
  if (one > cap_bytes)
    return fail(PLX_ERR_UNSUPPORTED,
                "%s: B * Hq = %lld needs %zu bytes of records even with one CTA; "
                "the fixed array holds %zu bytes (use plx_decode_fwd)",
                fn, static_cast<long long>(B) * Hq, one, cap_bytes);
  float *scratch = nullptr;
  cudaError_t e = plx::noalloc_scratch(&scratch);
  if (e != cudaSuccess) return cuda_fail(e, "plx_decode_fwd_noalloc: scratch address");
  // The default schedule, with as many CTAs as the array has records for.
  int nshare = plx_decode_default_nsplit(B, Hkv);
  while (nshare > 1 && plx_decode_workspace_bytes(B, Hq, Hkv, d, nshare) > cap_bytes) {
    const size_t per = plx_decode_workspace_bytes(B, Hq, Hkv, d, 2) -
                       plx_decode_workspace_bytes(B, Hq, Hkv, d, 1);
    const size_t over = plx_decode_workspace_bytes(B, Hq, Hkv, d, nshare) - cap_bytes;
    nshare -= static_cast<int>(std::min<size_t>(nshare - 1, (over + per - 1) / per));
  }
  return decode_bf16(fn, q, r, kcache, vcache, seqlens, out, nullptr, B, Hq, Hkv, d, nshare, true,
                     scratch, cap_bytes, stream);
}

plx_status plx_check_device_error(void *stream) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(e, "plx_check_device_error: stream");
  unsigned *w = plx::device_error_word();
  if (w == nullptr) return fail(PLX_ERR_CUDA, "plx_check_device_error: no error word");
  unsigned v = 0;
  e = cudaMemcpyAsync(&v, w, sizeof(v), cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaMemsetAsync(w, 0, sizeof(unsigned), st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(e, "plx_check_device_error: read");
  if (v & plx::kErrTimeout)
    return fail(PLX_ERR_DEVICE_TIMEOUT, "a bounded in-kernel wait ran out (error word 0x%x)", v);
  if (v & plx::kErrLayout)
    return fail(PLX_ERR_CUDA,
                "a kernel's dynamic shared memory was not 1024-byte aligned; it did no work "
                "(error word 0x%x)",
                v);
  if (v & plx::kErrBounds)
    return fail(PLX_ERR_BOUNDS,
                "a device-side bounds check failed; the access was skipped and the outputs "
                "are undefined (error word 0x%x)",
                v);
  if (v & plx::kErrBadInput)
    return fail(PLX_ERR_INVALID_ARG,
                "a kernel found device-side inputs out of range (decode: seqlens sum to 2^30 "
                "tokens or more); its outputs are undefined (error word 0x%x)",
                v);
  return PLX_OK;
}

plx_status plx_debug_timeout_probe(long long limit_cycles, void *stream) {
  if (limit_cycles < 0 || limit_cycles > (1LL << 32))
    return fail(PLX_ERR_INVALID_ARG, "plx_debug_timeout_probe: limit out of range");
  return finish_launch(plx::launch_timeout_probe(limit_cycles, plx::device_error_word(),
                                                 static_cast<cudaStream_t>(stream)),
                       "plx_debug_timeout_probe");
}

const char *plx_status_string(plx_status s) {
  switch (s) {
    case PLX_OK: return "ok";
    case PLX_ERR_INVALID_ARG: return "invalid argument";
    case PLX_ERR_UNSUPPORTED: return "unsupported configuration";
    case PLX_ERR_CUDA: return "CUDA error";
    case PLX_ERR_DEVICE_TIMEOUT: return "device wait timed out";
    case PLX_ERR_BOUNDS: return "device bounds check failed";
    default: return "unknown status";
  }
}

const char *plx_last_error_message(void) { return g_msg; }

}  // extern "C"
