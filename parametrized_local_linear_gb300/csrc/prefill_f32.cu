// Causal Parallax prefill in fp32 on the CUDA cores.
//
// One warp per query row; lane l owns head dims l, l + 32, ... . The keys are
// streamed once in order with the online-softmax recurrence of the pages'
// FlashAttention-compatible streaming algorithm ("Parallax: parametrized local
// linear attention for language modeling", section "Hardware-aware
// algorithm"), carrying four running quantities that share one running max m:
//   l  = sum_j e^{s_j - m}              (softmax denominator)
//   sg = sum_j e^{s_j - m} t_j           (t_j = rho_i . k_j)
//   a1 = sum_j e^{s_j - m} v_j           (-> O1 = a1 / l = o^SA)
//   a2 = sum_j e^{s_j - m} t_j v_j       (-> O2 = a2 / l)
// and finishing with o = O1 - O2 + O1 * (sg / l), which equals
// o^SA - Sigma_KV rho (section "Core mechanism") exactly in real arithmetic.
// Everything stays in fp32 with accurate expf/logf: this path exists for
// parity at 1e-5 relative error, not for speed.
#include <math.h>

#include "plx_internal.h"

namespace plx {
namespace {

constexpr int kRowsPerBlock = 8;

template <int D>
__global__ void __launch_bounds__(32 * kRowsPerBlock)
    prefill_f32_kernel(const float *__restrict__ q, const float *__restrict__ k,
                       const float *__restrict__ v, const float *__restrict__ r,
                       float *__restrict__ out, float *__restrict__ lse, int Hq, int Hkv, int L,
                       float tau) {
  constexpr int E = D / 32;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int i = blockIdx.x * kRowsPerBlock + warp;
  const int h = blockIdx.y, b = blockIdx.z;
  if (i >= L) return;
  const int g = h / (Hq / Hkv);
  const size_t qrow = ((static_cast<size_t>(b) * Hq + h) * L + i) * D;
  const float *kb = k + (static_cast<size_t>(b) * Hkv + g) * L * D;
  const float *vb = v + (static_cast<size_t>(b) * Hkv + g) * L * D;

  float qv[E], rv[E], a1[E], a2[E];
#pragma unroll
  for (int e = 0; e < E; ++e) {
    qv[e] = q[qrow + lane + 32 * e];
    rv[e] = r[qrow + lane + 32 * e];
    a1[e] = 0.f;
    a2[e] = 0.f;
  }
  float m = -INFINITY, l = 0.f, sg = 0.f;
  for (int j = 0; j <= i; ++j) {
    const float *kj = kb + static_cast<size_t>(j) * D;
    float s = 0.f, t = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const float kk = kj[lane + 32 * e];
      s = fmaf(qv[e], kk, s);
      t = fmaf(rv[e], kk, t);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      s += __shfl_xor_sync(0xffffffffu, s, o);
      t += __shfl_xor_sync(0xffffffffu, t, o);
    }
    s *= tau;
    const float mn = fmaxf(m, s);
    const float alpha = expf(m - mn);  // m = -inf on the first key: alpha = 0
    const float p = expf(s - mn);
    const float pt = p * t;
    l = fmaf(l, alpha, p);
    sg = fmaf(sg, alpha, pt);
    const float *vj = vb + static_cast<size_t>(j) * D;
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const float vv = vj[lane + 32 * e];
      a1[e] = fmaf(a1[e], alpha, p * vv);
      a2[e] = fmaf(a2[e], alpha, pt * vv);
    }
    m = mn;
  }
  const float inv = 1.f / l;
  const float sfac = sg * inv;
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const float o1 = a1[e] * inv, o2 = a2[e] * inv;
    out[qrow + lane + 32 * e] = o1 - o2 + o1 * sfac;
  }
  if (lse != nullptr && lane == 0)
    lse[(static_cast<size_t>(b) * Hq + h) * L + i] = m + logf(l);
}

}  // namespace

cudaError_t launch_prefill_f32(const float *q, const float *k, const float *v, const float *r,
                               float *out, float *lse, int B, int Hq, int Hkv, int L, int d,
                               unsigned * /*err*/, cudaStream_t stream) {
  dim3 grid((L + kRowsPerBlock - 1) / kRowsPerBlock, Hq, B);
  dim3 block(32 * kRowsPerBlock);
  const float tau = 1.0f / sqrtf(static_cast<float>(d));
  if (d == 64)
    prefill_f32_kernel<64><<<grid, block, 0, stream>>>(q, k, v, r, out, lse, Hq, Hkv, L, tau);
  else
    prefill_f32_kernel<128><<<grid, block, 0, stream>>>(q, k, v, r, out, lse, Hq, Hkv, L, tau);
  return cudaGetLastError();
}

}  // namespace plx
