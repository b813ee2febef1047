// Parallax decode: split-KV streaming over a packed bf16 KV cache, then a
// log-sum-exp combine of the per-split partial results.
//
// The method ("Parallax: parametrized local linear attention for language
// modeling", sections "Core mechanism" and "Hardware-aware algorithm") adds a
// covariance branch to softmax attention that reads the same KV stream; the
// pages' decode kernel therefore computes q.k and rho.k in the same tensor-core
// instructions so the cache is read from HBM once for both branches. This
// kernel does the same on sm_103a with warp-level mma.sync:
//
//   CTA (split s, kv head g, sequence b), 4 consumer warps + 1 producer warp.
//   Producer: one thread issues tiled TMA loads of 16-token x 64-dim boxes of
//     the K and V cache (3-D tensor maps over [tokens, Hkv, d]) into a ring of
//     8 shared-memory stages, 128-byte swizzled so ldmatrix is bank-conflict
//     free; completion is counted in bytes on per-stage mbarriers. Four 2 KB
//     requests move an 8 KB stage (per-row 256-byte copies were limited by
//     the TMA request rate).
//   Consumers: stages are dealt round-robin to the 4 warps, two per warp. For each 16 keys
//     one m16n8k16 product gives all four dot-product families at once: A rows
//     0..G-1 hold the G query heads' q, rows 8..8+G-1 their probes r, so the
//     accumulator row g is the score s = q.k and row g + 8 is t = r.k for the
//     same key in the same thread. P and P*T then form the A operand of the
//     value product (rows g: P -> O1, rows g + 8: P*T -> O2), again in
//     registers, with V^T read by ldmatrix.trans.
//   Each warp runs the online-softmax recurrence (running max m, denominator
//   l, sigma = sum p t, O1 and O2 accumulators, all rescaled together); the
//   warps are merged in shared memory and the CTA writes one partial record
//   per query head: (O1/l, O2/l, sigma/l, log2-sum-exp) in fp32.
//
// The combine kernel merges the records of a (sequence, head) with weights
// 2^(lse_s - max) and only then forms o = O1 - O2 + O1 * s. Combining final
// per-split outputs would be wrong: O1 * s is bilinear in the partial sums.
#include <math.h>

#include <mutex>

#include "plx_device.cuh"
#include "plx_internal.h"

namespace plx {
namespace {

constexpr int D = 128;
constexpr int KT = 16;                        // keys per stage (one TMA box row count)
constexpr int NCW = 4;                        // consumer warps
// Tile t goes to warp t % NCW and stage t % NST. NST is a multiple of NCW, so
// a stage is only ever consumed by one warp, which has itself consumed the
// stage's previous phase before it waits on the next one: a parity wait can
// never be two phases ahead (which it could not tell apart).
constexpr int NST = 2 * NCW;                  // stages in the ring
constexpr int HALF = KT * 128;                // one 64-dim half of KT rows, 128-byte swizzled
constexpr int STAGE_BYTES = 4 * HALF;         // K half 0, K half 1, V half 0, V half 1
constexpr int OFF_BAR = NST * STAGE_BYTES;    // 65536
static_assert(NST % NCW == 0, "each stage must belong to one consumer warp");
constexpr int SMEM_BYTES = OFF_BAR + 2 * NST * 8 + 16 + 1024;  // + alignment slack
constexpr int REC = 2 * D + 2;                // floats per partial record
constexpr int THREADS = 32 * (NCW + 1);

struct DecodeArgs {
  const __nv_bfloat16 *q, *r;
  const int *seqlens;
  float *ws;
  int B, Hq, Hkv, G, nsplit;
  float scale_log2;  // log2(e) / sqrt(d)
  unsigned *err;
};

// Byte offset of 16-byte chunk c (0..15 over the 128 dims) of row `row` in a
// stage half pair laid out by TMA with the 128-byte swizzle.
__device__ __forceinline__ uint32_t swz(int row, int c) {
  return (c >> 3) * HALF + row * 128 + ((((c & 7) ^ (row & 7))) << 4);
}

__global__ void __launch_bounds__(THREADS)
    decode_split_kernel(const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_v, const DecodeArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + OFF_BAR);
  uint64_t *empty = full + NST;
  volatile int *abort_flag = reinterpret_cast<volatile int *>(empty + NST);

  // kv heads vary fastest across the grid, so the CTAs that run side by side
  // read the same token range of neighbouring heads (adjacent 256-byte rows
  // of the cache): +1.5% on the ragged batch.
  const int kvh = blockIdx.x, split = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int len = a.seqlens[b];
  const int lo = static_cast<int>((static_cast<long long>(len) * split + a.nsplit - 1) / a.nsplit);
  const int hi =
      static_cast<int>((static_cast<long long>(len) * (split + 1) + a.nsplit - 1) / a.nsplit);
  const int nkeys = hi - lo;
  const int ntiles = (nkeys + KT - 1) / KT;

  if (threadIdx.x == 0) {
    for (int s = 0; s < NST; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), 1);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  const Abort ab{abort_flag, a.err};

  // Tile t covers keys [lo + KT t, min(lo + KT (t + 1), hi)). Its TMA box of KT
  // tokens starts at token min(off + lo + KT t, off + hi - KT), so the box
  // never reaches past the split's last key (and so never past the cache);
  // rows in front of the tile's first key (`skip` of them: keys of the
  // previous tile, or zero fill before token 0) are masked by the consumer.
  if (warp == NCW) {
    // ------------------------------------------------------------ producer
    long long off = 0;
    for (int i = lane; i < b; i += 32) off += a.seqlens[i];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) off += __shfl_xor_sync(0xffffffffu, off, o);
    if (lane == 0) {
      prefetch_tensormap(&tm_k);
      prefetch_tensormap(&tm_v);
      const int first = static_cast<int>(off) + lo, last = static_cast<int>(off) + hi;
      int issued = 0;
      for (int t = 0; t < ntiles; ++t) {
        const int st = t % NST;
        if (t >= NST && !mbar_wait(smem_u32(&empty[st]), ((t / NST) - 1) & 1, ab)) break;
        const uint32_t bar = smem_u32(&full[st]);
        mbar_arrive_expect_tx(bar, STAGE_BYTES);
        const int z = min(first + KT * t, last - KT);
        const uint32_t base = smem_u32(smem + st * STAGE_BYTES);
        tma_load_3d(base, &tm_k, 0, kvh, z, bar);
        tma_load_3d(base + HALF, &tm_k, 64, kvh, z, bar);
        tma_load_3d(base + 2 * HALF, &tm_v, 0, kvh, z, bar);
        tma_load_3d(base + 3 * HALF, &tm_v, 64, kvh, z, bar);
        issued = t + 1;
      }
      if (ab.raised()) {
        // Let this thread's own copies land before the CTA exits.
        for (int t = max(0, issued - NST); t < issued; ++t)
          mbar_wait_drain(smem_u32(&full[t % NST]), (t / NST) & 1);
      }
    }
  }

  // ------------------------------------------------------------ consumers
  const int g = lane >> 2, tq = lane & 3;
  float acc[16][4];
  float m = -INFINITY, l = 0.f, sg = 0.f;
#pragma unroll
  for (int i = 0; i < 16; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;

  if (warp < NCW) {
    uint32_t qa[8][4];
    {
      const bool live = g < a.G;
      const size_t hrow = (static_cast<size_t>(b) * a.Hq + kvh * a.G + (live ? g : 0)) * D;
      const uint32_t *qr = reinterpret_cast<const uint32_t *>(a.q + hrow);
      const uint32_t *rr = reinterpret_cast<const uint32_t *>(a.r + hrow);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        qa[kk][0] = live ? qr[8 * kk + tq] : 0u;
        qa[kk][1] = live ? rr[8 * kk + tq] : 0u;
        qa[kk][2] = live ? qr[8 * kk + 4 + tq] : 0u;
        qa[kk][3] = live ? rr[8 * kk + 4 + tq] : 0u;
      }
    }
    for (int t = warp; t < ntiles; t += NCW) {
      const int st = t % NST;
      bool ok = true;
      if (lane == 0) ok = mbar_wait(smem_u32(&full[st]), (t / NST) & 1, ab);
      if (!__shfl_sync(0xffffffffu, ok, 0)) break;
      const uint32_t kb = smem_u32(smem + st * STAGE_BYTES);
      const uint32_t vb = kb + 2 * HALF;
      // Rows [0, skip) of the box precede this tile's first key.
      const int skip = (lo + KT * t) - min(lo + KT * t, hi - KT);
#pragma unroll
      for (int half = 0; half < KT / 16; ++half) {
        if (half * 16 + 15 < skip) continue;
        float c[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
        const int krow = half * 16 + (lane >> 4) * 8 + (lane & 7);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          uint32_t b0, b1, b2, b3;
          ldsm_x4(kb + swz(krow, 2 * kk + ((lane >> 3) & 1)), b0, b1, b2, b3);
          mma_bf16_16816(c[0], qa[kk], b0, b1);
          mma_bf16_16816(c[1], qa[kk], b2, b3);
        }
        // c[n][0..1]: s for box rows half*16 + 8n + 2tq + {0,1}; c[n][2..3]: t for the same rows.
        float s[2][2];
        float mx = -INFINITY;
#pragma unroll
        for (int n = 0; n < 2; ++n)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int row = half * 16 + 8 * n + 2 * tq + e;
            s[n][e] = row >= skip ? c[n][e] * a.scale_log2 : -INFINITY;
            mx = fmaxf(mx, s[n][e]);
          }
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
        const float mn = fmaxf(m, mx);
        const float msub = mn == -INFINITY ? 0.f : mn;
        const float alpha = fast_exp2(m - msub);  // m = -inf: 0
        float p[2][2], pt[2][2], ps = 0.f, pts = 0.f;
#pragma unroll
        for (int n = 0; n < 2; ++n)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            p[n][e] = fast_exp2(s[n][e] - msub);
            pt[n][e] = p[n][e] * c[n][2 + e];
            ps += p[n][e];
            pts += pt[n][e];
          }
        l = fmaf(l, alpha, ps);
        sg = fmaf(sg, alpha, pts);
        m = mn;
        if (__any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            acc[i][0] *= alpha; acc[i][1] *= alpha; acc[i][2] *= alpha; acc[i][3] *= alpha;
          }
        }
        const uint32_t pa[4] = {pack_bf16x2(p[0][0], p[0][1]), pack_bf16x2(pt[0][0], pt[0][1]),
                                pack_bf16x2(p[1][0], p[1][1]), pack_bf16x2(pt[1][0], pt[1][1])};
        const int vrow = half * 16 + ((lane >> 3) & 1) * 8 + (lane & 7);
#pragma unroll
        for (int nd = 0; nd < 8; ++nd) {
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t(vb + swz(vrow, 2 * nd + (lane >> 4)), b0, b1, b2, b3);
          mma_bf16_16816(acc[2 * nd], pa, b0, b1);
          mma_bf16_16816(acc[2 * nd + 1], pa, b2, b3);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&empty[st]));
    }
    l += __shfl_xor_sync(0xffffffffu, l, 1);
    l += __shfl_xor_sync(0xffffffffu, l, 2);
    sg += __shfl_xor_sync(0xffffffffu, sg, 1);
    sg += __shfl_xor_sync(0xffffffffu, sg, 2);
  }

  // ------------------------------------------------------------ merge warps
  __syncthreads();  // every stage is consumed (or the CTA aborted): reuse them
  float *red = reinterpret_cast<float *>(smem);          // [NCW][2G][D]
  float *mls = red + NCW * 2 * a.G * D;                   // [NCW][G][3]
  if (warp < NCW && g < a.G) {
    float *o1 = red + (warp * 2 * a.G + g) * D;
    float *o2 = red + (warp * 2 * a.G + a.G + g) * D;
#pragma unroll
    for (int nd = 0; nd < 16; ++nd) {
      o1[8 * nd + 2 * tq] = acc[nd][0];
      o1[8 * nd + 2 * tq + 1] = acc[nd][1];
      o2[8 * nd + 2 * tq] = acc[nd][2];
      o2[8 * nd + 2 * tq + 1] = acc[nd][3];
    }
    if (tq == 0) {
      mls[(warp * a.G + g) * 3 + 0] = m;
      mls[(warp * a.G + g) * 3 + 1] = l;
      mls[(warp * a.G + g) * 3 + 2] = sg;
    }
  }
  __syncthreads();
  if (threadIdx.x < D) {
    const int dim = threadIdx.x;
    for (int gh = 0; gh < a.G; ++gh) {
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < NCW; ++w) M = fmaxf(M, mls[(w * a.G + gh) * 3]);
      float *rec = a.ws + ((static_cast<size_t>(b) * a.Hq + kvh * a.G + gh) * a.nsplit + split) * REC;
      if (M == -INFINITY || ab.raised()) {
        rec[dim] = 0.f;
        rec[D + dim] = 0.f;
        if (dim == 0) {
          rec[2 * D] = 0.f;
          rec[2 * D + 1] = -INFINITY;
        }
        continue;
      }
      float L = 0.f, S = 0.f, O1 = 0.f, O2 = 0.f;
#pragma unroll
      for (int w = 0; w < NCW; ++w) {
        const float f = fast_exp2(mls[(w * a.G + gh) * 3] - M);
        L = fmaf(f, mls[(w * a.G + gh) * 3 + 1], L);
        S = fmaf(f, mls[(w * a.G + gh) * 3 + 2], S);
        O1 = fmaf(f, red[(w * 2 * a.G + gh) * D + dim], O1);
        O2 = fmaf(f, red[(w * 2 * a.G + a.G + gh) * D + dim], O2);
      }
      const float inv = 1.f / L;
      rec[dim] = O1 * inv;
      rec[D + dim] = O2 * inv;
      if (dim == 0) {
        rec[2 * D] = S * inv;
        rec[2 * D + 1] = M + log2f(L);
      }
    }
  }
}

// One block of D threads per (sequence, query head): merge the splits.
__global__ void __launch_bounds__(D) decode_combine_kernel(const float *__restrict__ ws,
                                                          __nv_bfloat16 *__restrict__ out,
                                                          float *__restrict__ cor, int nsplit) {
  const int bh = blockIdx.x, dim = threadIdx.x;
  const float *rec = ws + static_cast<size_t>(bh) * nsplit * REC;
  float M = -INFINITY;
  for (int s = 0; s < nsplit; ++s) M = fmaxf(M, rec[s * REC + 2 * D + 1]);
  float o = 0.f, c = 0.f;
  if (M != -INFINITY) {
    float W = 0.f, o1 = 0.f, o2 = 0.f, sf = 0.f;
    for (int s = 0; s < nsplit; ++s) {
      const float lse = rec[s * REC + 2 * D + 1];
      const float w = exp2f(lse - M);  // empty split: lse = -inf, w = 0
      W += w;
      o1 = fmaf(w, rec[s * REC + dim], o1);
      o2 = fmaf(w, rec[s * REC + D + dim], o2);
      sf = fmaf(w, rec[s * REC + 2 * D], sf);
    }
    const float inv = 1.f / W;
    o1 *= inv;
    o2 *= inv;
    sf *= inv;
    c = o2 - o1 * sf;  // the correction Sigma rho
    o = o1 - c;
  }
  out[static_cast<size_t>(bh) * D + dim] = __float2bfloat16_rn(o);
  if (cor != nullptr) {
    // |correction| / |o| over the head's d values: warp sums, then 4 warps.
    __shared__ float part[2][D / 32];
    float csq = c * c, osq = o * o;
#pragma unroll
    for (int sh = 16; sh > 0; sh >>= 1) {
      csq += __shfl_xor_sync(0xffffffffu, csq, sh);
      osq += __shfl_xor_sync(0xffffffffu, osq, sh);
    }
    if ((dim & 31) == 0) {
      part[0][dim >> 5] = csq;
      part[1][dim >> 5] = osq;
    }
    __syncthreads();
    if (dim == 0) {
      float cs = 0.f, os = 0.f;
#pragma unroll
      for (int w = 0; w < D / 32; ++w) {
        cs += part[0][w];
        os += part[1][w];
      }
      cor[bh] = os > 0.f ? sqrtf(cs) / sqrtf(os) : 0.f;
    }
  }
}

}  // namespace

cudaError_t launch_decode(const void *q, const void *r, const void *kcache, const void *vcache,
                          const int *seqlens, void *out, float *cor, int B, int Hq, int Hkv,
                          int nsplit, float *workspace, unsigned *err, cudaStream_t stream) {
  static thread_local int configured_device = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (configured_device != dev) {
    cudaError_t e = cudaFuncSetAttribute(decode_split_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) return e;
    configured_device = dev;
  }
  EncodeTiledFn enc = encode_tiled_fn();
  if (enc == nullptr) return cudaErrorInvalidValue;
  // The cache is [tokens, Hkv, d]. Its token count lives on the device, so the
  // map declares 2^30 tokens; every box the kernel requests lies inside the
  // tokens of its own sequence (or, for caches shorter than one box, starts
  // at a negative token and is zero-filled there).
  CUtensorMap mk, mv;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(Hkv),
                              static_cast<cuuint64_t>(1) << 30};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2,
                                 static_cast<cuuint64_t>(Hkv) * D * 2};
  const cuuint32_t box[3] = {64, 1, KT};
  const cuuint32_t estr[3] = {1, 1, 1};
  for (int i = 0; i < 2; ++i) {
    if (enc(i == 0 ? &mk : &mv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
            const_cast<void *>(i == 0 ? kcache : vcache), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  DecodeArgs a;
  a.q = static_cast<const __nv_bfloat16 *>(q);
  a.r = static_cast<const __nv_bfloat16 *>(r);
  a.seqlens = seqlens;
  a.ws = workspace;
  a.B = B;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.G = Hq / Hkv;
  a.nsplit = nsplit;
  a.scale_log2 = 1.4426950408889634f / sqrtf(static_cast<float>(D));
  a.err = err;
  decode_split_kernel<<<dim3(Hkv, nsplit, B), THREADS, SMEM_BYTES, stream>>>(mk, mv, a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  decode_combine_kernel<<<B * Hq, D, 0, stream>>>(workspace, static_cast<__nv_bfloat16 *>(out),
                                                  cor, nsplit);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Decode without any allocation. Some callers cannot allocate device memory
// at call time: code whose device memory belongs to an allocator that must
// not be bypassed, a host thread that must not take the driver's allocation
// locks, or an embedding that hands this library only its own input and
// output buffers. For them the
// split records live in one fixed array below, reserved when the library is
// loaded onto a device and held by every device that loads it until the
// process exits. Its address is resolved with cudaGetSymbolAddress once per
// device, on the first call on that device (make that first call before any
// stream capture). Calls that overlap on the GPU share the array and race;
// serialise them (one stream, or events). Nothing in it needs clearing between
// calls: each call's split kernel writes every record that its combine kernel
// then reads.
static __device__ __align__(256) float g_decode_noalloc_scratch[kNoAllocScratchFloats];

namespace {
std::mutex g_noalloc_mu;
float *g_noalloc_ptr[64] = {};
}  // namespace

cudaError_t noalloc_scratch(float **ptr) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (g_noalloc_ptr[dev] == nullptr) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_decode_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_noalloc_ptr[dev] = static_cast<float *>(p);
  }
  *ptr = g_noalloc_ptr[dev];
  return cudaSuccess;
}

}  // namespace plx
