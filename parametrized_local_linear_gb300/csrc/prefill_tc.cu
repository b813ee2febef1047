// Causal Parallax prefill on the 5th-generation tensor cores (tcgen05, TMEM,
// TMA), bf16 operands, fp32 accumulation, d = 128.
//
// Algorithm: the pages' FlashAttention-compatible streaming form ("Parallax:
// parametrized local linear attention for language modeling", section
// "Hardware-aware algorithm"), which for every key tile does four GEMMs on one
// K/V stream instead of softmax attention's two:
//   S = Q K^T,  T = R K^T,  O1 += P V,  O2 += (P o T) V,
// with P = exp(S/sqrt(d) - m) under one running max m shared by the
// denominator l, by sigma = rowsum(P o T) and by both accumulators, and
// finishes o = (O1 (1 + sigma / l) - O2) / l, i.e. o^SA - Sigma_KV rho
// (section "Core mechanism").
//
// One CTA owns 128 query rows of one (batch, head); 6 warps:
//   warp 0      TMA producer: Q and R once (128 x 128 each), then K_j, V_j
//               (64 keys x 128) into a 3-stage ring, 128-byte swizzled.
//   warp 1      TMEM allocator and single-thread UMMA issuer.
//   warps 2..5  softmax / epilogue: thread = query row = TMEM lane.
// Tensor memory (512 columns x 128 lanes, fp32):
//   [0,64) S_0  [64,128) T_0  [128,192) S_1  [192,256) T_1  (double buffered)
//   [256,384) O1              [384,512) O2
// The UMMA for tile j+1 (S, T into buffer (j+1)&1) runs while the softmax
// warps work on tile j. The softmax writes P and P o T as packed bf16 over
// the S columns of its buffer (S_x[0,32) = P, S_x[32,64) = P o T) and the value
// GEMMs read them straight from TMEM (A-from-TMEM form), V from shared memory
// (MN-major). Rescaling is lazy: the max used in the exponent only moves when
// a row's tile max exceeds it by more than 2^8, which keeps every quantity
// exact (they all share the stale max) and rarely touches O in TMEM.
#include <math.h>

#include "plx_device.cuh"
#include "plx_internal.h"

namespace plx {
namespace {

constexpr int D = 128;
constexpr int BM = 128;                       // query rows per CTA
constexpr int BN = 64;                        // keys per tile
constexpr int NST = 3;                        // K/V stages
constexpr int HALF_Q = BM * 64 * 2;           // 16 KB: 128 rows x 64 dims
constexpr int HALF_KV = BN * 64 * 2;          // 8 KB: 64 rows x 64 dims
constexpr int TILE_KV = 2 * HALF_KV;          // 16 KB
constexpr int STAGE_BYTES = 2 * TILE_KV;      // K then V
constexpr int OFF_Q = 0;
constexpr int OFF_R = 2 * HALF_Q;
constexpr int OFF_KV = 4 * HALF_Q;            // 65536
constexpr int OFF_BAR = OFF_KV + NST * STAGE_BYTES;  // 163840
constexpr int NBAR = 1 + 2 * NST + 2 + 2 + 1 + 1;
constexpr int SMEM_BYTES = OFF_BAR + NBAR * 8 + 16 + 1024;  // + alignment slack
constexpr int THREADS = 192;
constexpr uint32_t COL_S0 = 0, COL_S1 = 128, COL_T = 64, COL_O1 = 256, COL_O2 = 384;
constexpr float kRescaleThreshold = 8.0f;     // log2 units

struct PrefillArgs {
  float *lse;
  int Hq, Hkv, L, B, nqt;
  float scale_log2;  // log2(e) / sqrt(d)
  unsigned *err;
};

__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

__global__ void __launch_bounds__(THREADS, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_r,
                      const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                      const __grid_constant__ CUtensorMap tm_o, const PrefillArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + OFF_BAR);
  uint64_t *q_full = bars;
  uint64_t *kv_full = bars + 1;
  uint64_t *kv_empty = bars + 1 + NST;
  uint64_t *st_full = bars + 1 + 2 * NST;
  uint64_t *p_full = st_full + 2;
  uint64_t *pv_done = p_full + 2;
  uint64_t *mma_drain = pv_done + 1;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + NBAR);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // Longest (most keys) query tiles first.
  const int per_qt = a.Hq * a.B;
  const int qt = a.nqt - 1 - static_cast<int>(blockIdx.x) / per_qt;
  const int rem = static_cast<int>(blockIdx.x) % per_qt;
  const int h = rem % a.Hq, b = rem / a.Hq;
  const int q0 = qt * BM;
  const int kv_end = min(q0 + BM, a.L);
  const int ntiles = (kv_end + BN - 1) / BN;
  const int zq = b * a.Hq + h;
  const int zk = b * a.Hkv + h / (a.Hq / a.Hkv);

  if (threadIdx.x == 0) {
    mbar_init(smem_u32(q_full), 1);
    for (int s = 0; s < NST; ++s) {
      mbar_init(smem_u32(&kv_full[s]), 1);
      mbar_init(smem_u32(&kv_empty[s]), 1);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(smem_u32(&st_full[x]), 1);
      mbar_init(smem_u32(&p_full[x]), 128);
    }
    mbar_init(smem_u32(pv_done), 1);
    mbar_init(smem_u32(mma_drain), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tensormap(&tm_q);
    prefetch_tensormap(&tm_r);
    prefetch_tensormap(&tm_k);
    prefetch_tensormap(&tm_v);
    prefetch_tensormap(&tm_o);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;
  const Abort ab{abort_flag, a.err};

  if (warp == 0) {
    if (lane == 0) {
      // ---------------------------------------------------------- producer
      const uint32_t qb = smem_u32(q_full);
      mbar_arrive_expect_tx(qb, 4 * HALF_Q);
      tma_load_3d(smem_u32(smem + OFF_Q), &tm_q, 0, q0, zq, qb);
      tma_load_3d(smem_u32(smem + OFF_Q + HALF_Q), &tm_q, 64, q0, zq, qb);
      tma_load_3d(smem_u32(smem + OFF_R), &tm_r, 0, q0, zq, qb);
      tma_load_3d(smem_u32(smem + OFF_R + HALF_Q), &tm_r, 64, q0, zq, qb);
      int issued = 0;
      for (int j = 0; j < ntiles; ++j) {
        const int st = j % NST;
        if (j >= NST && !mbar_wait(smem_u32(&kv_empty[st]), ((j / NST) - 1) & 1, ab)) break;
        const uint32_t fb = smem_u32(&kv_full[st]);
        mbar_arrive_expect_tx(fb, STAGE_BYTES);
        const uint32_t base = smem_u32(smem + OFF_KV + st * STAGE_BYTES);
        tma_load_3d(base, &tm_k, 0, j * BN, zk, fb);
        tma_load_3d(base + HALF_KV, &tm_k, 64, j * BN, zk, fb);
        tma_load_3d(base + TILE_KV, &tm_v, 0, j * BN, zk, fb);
        tma_load_3d(base + TILE_KV + HALF_KV, &tm_v, 64, j * BN, zk, fb);
        issued = j + 1;
      }
      if (ab.raised()) {
        mbar_wait_drain(qb, 0);
        for (int j = max(0, issued - NST); j < issued; ++j)
          mbar_wait_drain(smem_u32(&kv_full[j % NST]), (j / NST) & 1);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------------------------------------------------- UMMA issuer
      constexpr uint32_t idesc_st = idesc_bf16_f32(BM, BN, 0);
      constexpr uint32_t idesc_pv = idesc_bf16_f32(BM, D, 1);
      const uint32_t sq = smem_u32(smem + OFF_Q), sr = smem_u32(smem + OFF_R);
      auto issue_st = [&](int j) -> bool {
        const int st = j % NST;
        if (!mbar_wait(smem_u32(&kv_full[st]), (j / NST) & 1, ab)) return false;
        tc_fence_after();
        const uint32_t kb = smem_u32(smem + OFF_KV + st * STAGE_BYTES);
        const uint32_t cs = tbase + ((j & 1) ? COL_S1 : COL_S0);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint32_t qo = (ks >> 2) * HALF_Q + (ks & 3) * 32;
          const uint32_t ko = (ks >> 2) * HALF_KV + (ks & 3) * 32;
          umma_ss(cs, smem_desc_sw128(sq + qo, 16, 1024), smem_desc_sw128(kb + ko, 16, 1024),
                  idesc_st, ks > 0);
        }
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint32_t qo = (ks >> 2) * HALF_Q + (ks & 3) * 32;
          const uint32_t ko = (ks >> 2) * HALF_KV + (ks & 3) * 32;
          umma_ss(cs + COL_T, smem_desc_sw128(sr + qo, 16, 1024),
                  smem_desc_sw128(kb + ko, 16, 1024), idesc_st, ks > 0);
        }
        umma_commit(smem_u32(&st_full[j & 1]));
        return true;
      };
      bool ok = mbar_wait(smem_u32(q_full), 0, ab);
      if (ok) {
        tc_fence_after();
        ok = issue_st(0);
      }
      for (int j = 0; ok && j < ntiles; ++j) {
        if (j + 1 < ntiles && !issue_st(j + 1)) break;
        if (!mbar_wait(smem_u32(&p_full[j & 1]), (j >> 1) & 1, ab)) break;
        tc_fence_after();
        const uint32_t vb = smem_u32(smem + OFF_KV + (j % NST) * STAGE_BYTES + TILE_KV);
        const uint32_t cp = tbase + ((j & 1) ? COL_S1 : COL_S0);
#pragma unroll
        for (int ks = 0; ks < BN / 16; ++ks)
          umma_ts(tbase + COL_O1, cp + ks * 8, smem_desc_sw128(vb + ks * 2048, HALF_KV, 1024),
                  idesc_pv, (j > 0 || ks > 0));
#pragma unroll
        for (int ks = 0; ks < BN / 16; ++ks)
          umma_ts(tbase + COL_O2, cp + 32 + ks * 8, smem_desc_sw128(vb + ks * 2048, HALF_KV, 1024),
                  idesc_pv, (j > 0 || ks > 0));
        umma_commit(smem_u32(pv_done));
        umma_commit(smem_u32(&kv_empty[j % NST]));
      }
      // Every UMMA this thread issued must finish before TMEM is released.
      umma_commit(smem_u32(mma_drain));
      mbar_wait_drain(smem_u32(mma_drain), 0);
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int qw = warp & 3;             // TMEM lane quarter this warp may touch
    const int row = qw * 32 + lane;      // query row within the tile
    const int grow = q0 + row;
    const uint32_t tl = tbase + (static_cast<uint32_t>(qw * 32) << 16);
    const float c = a.scale_log2;
    float m_used = -INFINITY, l = 0.f, sg = 0.f;
    bool ok = true;
    for (int j = 0; j < ntiles; ++j) {
      const int x = j & 1;
      ok = mbar_wait(smem_u32(&st_full[x]), (j >> 1) & 1, ab);
      if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      tc_fence_after();
      const uint32_t cs = tl + (x ? COL_S1 : COL_S0);
      float s[64], t[64];
      tmem_ld32(cs, *reinterpret_cast<float(*)[32]>(&s[0]));
      tmem_ld32(cs + 32, *reinterpret_cast<float(*)[32]>(&s[32]));
      tmem_ld32(cs + COL_T, *reinterpret_cast<float(*)[32]>(&t[0]));
      tmem_ld32(cs + COL_T + 32, *reinterpret_cast<float(*)[32]>(&t[32]));
      tmem_wait_ld();
      if (j * BN + BN - 1 > q0) {  // tile reaches the diagonal: causal mask
#pragma unroll
        for (int e = 0; e < BN; ++e)
          if (j * BN + e > grow) s[e] = -INFINITY;
      }
      float mt = -INFINITY;
#pragma unroll
      for (int e = 0; e < BN; ++e) mt = fmaxf(mt, s[e]);
      mt *= c;
      const bool need = mt > m_used + kRescaleThreshold;
      float alpha = 1.f;
      if (need) {
        alpha = fast_exp2(m_used - mt);  // m_used = -inf: 0
        l *= alpha;
        sg *= alpha;
        m_used = mt;
      }
      const float msub = m_used == -INFINITY ? 0.f : m_used;
      uint32_t pk[32], ptk[32];
#pragma unroll
      for (int e = 0; e < BN; e += 2) {
        const float p0 = fast_exp2(fmaf(s[e], c, -msub));
        const float p1 = fast_exp2(fmaf(s[e + 1], c, -msub));
        const float pt0 = p0 * t[e], pt1 = p1 * t[e + 1];
        l += p0 + p1;
        sg += pt0 + pt1;
        pk[e >> 1] = pack_bf16x2(p0, p1);
        ptk[e >> 1] = pack_bf16x2(pt0, pt1);
      }
      tmem_st16(cs, *reinterpret_cast<uint32_t(*)[16]>(&pk[0]));
      tmem_st16(cs + 16, *reinterpret_cast<uint32_t(*)[16]>(&pk[16]));
      tmem_st16(cs + 32, *reinterpret_cast<uint32_t(*)[16]>(&ptk[0]));
      tmem_st16(cs + 48, *reinterpret_cast<uint32_t(*)[16]>(&ptk[16]));
      tmem_wait_st();
      if (j > 0) {
        // The previous tile's value GEMMs must be done before O is touched
        // and before P of this tile is handed over.
        ok = mbar_wait(smem_u32(pv_done), (j - 1) & 1, ab);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        tc_fence_after();
        if (__any_sync(0xffffffffu, need)) {
#pragma unroll 1
          for (int part = 0; part < 8; ++part) {
            const uint32_t col = (part < 4 ? COL_O1 : COL_O2) + (part & 3) * 32;
            float o[32];
            tmem_ld32(tl + col, o);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] *= alpha;
            tmem_st32(tl + col, o);
          }
          tmem_wait_st();
        }
      }
      tc_fence_before();
      mbar_arrive(smem_u32(&p_full[x]));
    }
    if (ok) {
      ok = mbar_wait(smem_u32(pv_done), (ntiles - 1) & 1, ab);
      ok = __all_sync(0xffffffffu, ok);
    }
    uint8_t *so = smem + OFF_Q;  // Q is dead once every UMMA has finished
    if (ok) {
      tc_fence_after();
      const float inv = 1.f / l;
      const float g1 = (1.f + sg * inv) * inv;
#pragma unroll 1
      for (int part = 0; part < 4; ++part) {
        float o1[32], o2[32];
        tmem_ld32(tl + COL_O1 + part * 32, o1);
        tmem_ld32(tl + COL_O2 + part * 32, o2);
        tmem_wait_ld();
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 32; e += 2)
          pk[e >> 1] = pack_bf16x2(fmaf(o1[e], g1, -o2[e] * inv), fmaf(o1[e + 1], g1, -o2[e + 1] * inv));
        // 32 dims = four 16-byte chunks; 128-byte swizzle as the TMA store expects.
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int cc = part * 4 + u;
          uint8_t *dst = so + (cc >> 3) * HALF_Q + row * 128 + (((cc & 7) ^ (row & 7)) << 4);
          *reinterpret_cast<uint4 *>(dst) = make_uint4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
        }
      }
      if (a.lse != nullptr && grow < a.L)
        a.lse[static_cast<size_t>(zq) * a.L + grow] = (m_used + log2f(l)) * 0.6931471805599453f;
      fence_proxy_async_smem();
    }
    named_bar_sync(1, 128);
    if (warp == 2 && lane == 0 && !ab.raised()) {
      tma_store_3d(&tm_o, smem_u32(so), 0, q0, zq);
      tma_store_3d(&tm_o, smem_u32(so + HALF_Q), 64, q0, zq);
      bulk_commit_group();
      bulk_wait_group_all();
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
}

bool make_map(EncodeTiledFn enc, CUtensorMap *map, const void *ptr, int L, int heads, int box_rows) {
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(L),
                              static_cast<cuuint64_t>(heads)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2,
                                 static_cast<cuuint64_t>(L) * D * 2};
  const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(box_rows), 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(ptr), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_prefill_tc(const void *q, const void *k, const void *v, const void *r, void *out,
                              float *lse, int B, int Hq, int Hkv, int L, unsigned *err,
                              cudaStream_t stream) {
  static thread_local int configured_device = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (configured_device != dev) {
    cudaError_t e = cudaFuncSetAttribute(prefill_tc_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) return e;
    configured_device = dev;
  }
  EncodeTiledFn enc = encode_tiled_fn();
  if (enc == nullptr) return cudaErrorInvalidValue;
  CUtensorMap mq, mr, mk, mv, mo;
  if (!make_map(enc, &mq, q, L, B * Hq, BM) || !make_map(enc, &mr, r, L, B * Hq, BM) ||
      !make_map(enc, &mk, k, L, B * Hkv, BN) || !make_map(enc, &mv, v, L, B * Hkv, BN) ||
      !make_map(enc, &mo, out, L, B * Hq, BM))
    return cudaErrorInvalidValue;
  PrefillArgs a;
  a.lse = lse;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.L = L;
  a.B = B;
  a.nqt = (L + BM - 1) / BM;
  a.scale_log2 = 1.4426950408889634f / sqrtf(static_cast<float>(D));
  a.err = err;
  const unsigned grid = static_cast<unsigned>(a.nqt) * Hq * B;
  prefill_tc_kernel<<<grid, THREADS, SMEM_BYTES, stream>>>(mq, mr, mk, mv, mo, a);
  return cudaGetLastError();
}

}  // namespace plx
