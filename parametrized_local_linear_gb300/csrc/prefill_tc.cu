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
// One CTA owns 128 query rows of one (batch, head); 9 warps:
//   warp 0      TMA producer: Q and R once (128 x 128 each), then K_j and V_j
//               (64 keys x 128 each) into two 4-stage rings, 128-byte
//               swizzled. A K tile is released once the S and T UMMAs that
//               read it finish, a V tile once the value UMMAs finish.
//   warp 1      TMEM allocator; one thread issues O1 += P V.
//   warp 2      one thread issues O2 += (P o T) V.
//   warps 3..6  softmax / epilogue: thread = query row = TMEM lane.
//   warp 7      one thread issues S = Q K^T.
//   warp 8      one thread issues T = R K^T.
// Four issuing threads, because one thread cannot issue tcgen05.mma as fast
// as the tensor core retires these shapes (measured: 50-100 cycles per issue
// under load against 48-64 cycles of work per instruction). The value UMMAs,
// which sit on the critical path (softmax -> P V -> next softmax), have
// issuers of their own that respond at once; S and T of tile j + 2 overwrite
// P(j) and P o T(j) and therefore wait for the value UMMAs of tile j
// (pv_done), which leaves them two tiles of slack.
// Tensor memory (512 columns x 128 lanes, fp32):
//   [0,64) S_0  [64,128) T_0  [128,192) S_1  [192,256) T_1  (double buffered)
//   [256,384) O1              [384,512) O2
// The UMMAs for tile j+1 run while the softmax warps work on tile j. The
// softmax writes P and P o T as packed bf16 (S_x[0,32) = P, T_x[0,32) =
// P o T) and the value GEMMs read them straight from TMEM (A-from-TMEM
// form), V from shared memory (MN-major). Rescaling is
// lazy: the max used in the exponent only moves when a row's tile max
// exceeds it by more than 2^8, which keeps every quantity exact (they all
// share the stale max) and rarely touches O in TMEM.
#include <math.h>

#include "plx_device.cuh"
#include "plx_internal.h"

namespace plx {
namespace {

constexpr int D = 128;
constexpr int BM = 128;                       // query rows per CTA
constexpr int BN = 64;                        // keys per tile
constexpr int NST = 4;                        // stages per K / V ring
constexpr int HALF_Q = BM * 64 * 2;           // 16 KB: 128 rows x 64 dims
constexpr int HALF_KV = BN * 64 * 2;          // 8 KB: 64 rows x 64 dims
constexpr int TILE_KV = 2 * HALF_KV;          // 16 KB: one K or V tile
constexpr int OFF_Q = 0;
constexpr int OFF_R = 2 * HALF_Q;
constexpr int OFF_K = 4 * HALF_Q;             // 65536
constexpr int OFF_V = OFF_K + NST * TILE_KV;  // 131072
constexpr int OFF_BAR = OFF_V + NST * TILE_KV;  // 196608
constexpr int NBAR = 1 + 4 * NST + 2 + 2 + 2 + 4;
constexpr int SMEM_BYTES = OFF_BAR + NBAR * 8 + 16 + 1024;  // + alignment slack
constexpr int SM_WARP0 = 3;                   // first softmax warp
constexpr int THREADS = 32 * 9;
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
  uint64_t *k_full = bars + 1;
  uint64_t *k_empty = k_full + NST;
  uint64_t *v_full = k_empty + NST;
  uint64_t *v_empty = v_full + NST;
  uint64_t *st_full = v_empty + NST;   // [2]
  uint64_t *p_full = st_full + 2;      // [2]
  uint64_t *pv_done = p_full + 2;      // [2]: value UMMAs of the tiles using buffer x
  uint64_t *drain = pv_done + 2;       // [4]: one per issuing thread
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
      mbar_init(smem_u32(&k_full[s]), 1);
      mbar_init(smem_u32(&k_empty[s]), 2);
      mbar_init(smem_u32(&v_full[s]), 1);
      mbar_init(smem_u32(&v_empty[s]), 2);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(smem_u32(&st_full[x]), 2);
      mbar_init(smem_u32(&p_full[x]), 128);
      mbar_init(smem_u32(&pv_done[x]), 2);
    }
    for (int x = 0; x < 4; ++x) mbar_init(smem_u32(&drain[x]), 1);
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
      int k_issued = 0, v_issued = 0;
      for (int j = 0; j < ntiles; ++j) {
        const int st = j % NST;
        if (j >= NST && !mbar_wait(smem_u32(&k_empty[st]), ((j / NST) - 1) & 1, ab)) break;
        const uint32_t kf = smem_u32(&k_full[st]);
        mbar_arrive_expect_tx(kf, TILE_KV);
        const uint32_t kb = smem_u32(smem + OFF_K + st * TILE_KV);
        tma_load_3d(kb, &tm_k, 0, j * BN, zk, kf);
        tma_load_3d(kb + HALF_KV, &tm_k, 64, j * BN, zk, kf);
        k_issued = j + 1;
        if (j >= NST && !mbar_wait(smem_u32(&v_empty[st]), ((j / NST) - 1) & 1, ab)) break;
        const uint32_t vf = smem_u32(&v_full[st]);
        mbar_arrive_expect_tx(vf, TILE_KV);
        const uint32_t vb = smem_u32(smem + OFF_V + st * TILE_KV);
        tma_load_3d(vb, &tm_v, 0, j * BN, zk, vf);
        tma_load_3d(vb + HALF_KV, &tm_v, 64, j * BN, zk, vf);
        v_issued = j + 1;
      }
      if (ab.raised()) {
        // Let this thread's own copies land before the CTA exits.
        mbar_wait_drain(qb, 0);
        for (int j = max(0, k_issued - NST); j < k_issued; ++j)
          mbar_wait_drain(smem_u32(&k_full[j % NST]), (j / NST) & 1);
        for (int j = max(0, v_issued - NST); j < v_issued; ++j)
          mbar_wait_drain(smem_u32(&v_full[j % NST]), (j / NST) & 1);
      }
    }
  } else if (warp == 1 || warp == 2) {
    if (lane == 0) {
      // ---------------------------------------------------------- value UMMAs
      // Warp 1: O1 += P V (P over S); warp 2: O2 += (P o T) V (over T).
      const bool is_o1 = warp == 1;
      constexpr uint32_t idesc_pv = idesc_bf16_f32(BM, D, 1);
      const uint64_t vdesc0 = smem_desc_sw128(smem_u32(smem + OFF_V), HALF_KV, 1024);
      const uint32_t col_off = is_o1 ? 0u : COL_T;
      const uint32_t dout = tbase + (is_o1 ? COL_O1 : COL_O2);
      for (int j = 0; j < ntiles; ++j) {
        const int x = j & 1, st = j % NST;
        if (!mbar_wait(smem_u32(&p_full[x]), (j >> 1) & 1, ab)) break;
        if (!mbar_wait(smem_u32(&v_full[st]), (j / NST) & 1, ab)) break;
        tc_fence_after();
        const uint64_t vdesc = vdesc0 + st * (TILE_KV >> 4);
        const uint32_t ap = tbase + (x ? COL_S1 : COL_S0) + col_off;
#pragma unroll
        for (int ks = 0; ks < BN / 16; ++ks)
          umma_ts(dout, ap + ks * 8, vdesc + ks * (2048 >> 4), idesc_pv, (j > 0 || ks > 0));
        umma_commit(smem_u32(&pv_done[x]));
        umma_commit(smem_u32(&v_empty[st]));
      }
      // Every UMMA this thread issued must finish before TMEM is released.
      umma_commit(smem_u32(&drain[is_o1 ? 0 : 1]));
      mbar_wait_drain(smem_u32(&drain[is_o1 ? 0 : 1]), 0);
    }
  } else if (warp == 7 || warp == 8) {
    if (lane == 0) {
      // ---------------------------------------------------------- score UMMAs
      // Warp 7: S = Q K^T; warp 8: T = R K^T. Descriptors are built once; a K
      // step only adds a constant to the start-address field (16-byte units,
      // never carrying out of its 14 bits since shared memory is below 256 KB).
      const bool is_s = warp == 7;
      constexpr uint32_t idesc_st = idesc_bf16_f32(BM, BN, 0);
      const uint64_t adesc = smem_desc_sw128(smem_u32(smem + (is_s ? OFF_Q : OFF_R)), 16, 1024);
      const uint64_t kdesc0 = smem_desc_sw128(smem_u32(smem + OFF_K), 16, 1024);
      const uint32_t col_off = is_s ? 0u : COL_T;
      bool ok = mbar_wait(smem_u32(q_full), 0, ab);
      for (int j = 0; ok && j < ntiles; ++j) {
        const int x = j & 1, st = j % NST;
        // Buffer x still holds P / P o T of tile j - 2 until its value UMMAs finish.
        if (j >= 2 && !mbar_wait(smem_u32(&pv_done[x]), ((j - 2) >> 1) & 1, ab)) break;
        if (!mbar_wait(smem_u32(&k_full[st]), (j / NST) & 1, ab)) break;
        tc_fence_after();
        const uint64_t kdesc = kdesc0 + st * (TILE_KV >> 4);
        const uint32_t d = tbase + (x ? COL_S1 : COL_S0) + col_off;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks)
          umma_ss(d, adesc + (ks >> 2) * (HALF_Q >> 4) + (ks & 3) * 2,
                  kdesc + (ks >> 2) * (HALF_KV >> 4) + (ks & 3) * 2, idesc_st, ks > 0);
        umma_commit(smem_u32(&st_full[x]));
        umma_commit(smem_u32(&k_empty[st]));
      }
      umma_commit(smem_u32(&drain[is_s ? 2 : 3]));
      mbar_wait_drain(smem_u32(&drain[is_s ? 2 : 3]), 0);
    }
  } else if (warp >= SM_WARP0 && warp < SM_WARP0 + 4) {
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
      float s[64];
      tmem_ld32(cs, *reinterpret_cast<float(*)[32]>(&s[0]));
      tmem_ld32(cs + 32, *reinterpret_cast<float(*)[32]>(&s[32]));
      tmem_wait_ld();
      if (j * BN + BN - 1 > q0) {  // tile reaches the diagonal: causal mask
#pragma unroll
        for (int e = 0; e < BN; ++e)
          if (j * BN + e > grow) s[e] = -INFINITY;
      }
      // Row max: 8 independent chains of 3-input max, then a tree.
      float mx8[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) mx8[e] = fmaxf(s[2 * e], s[2 * e + 1]);
#pragma unroll
      for (int e = 16; e < BN; e += 2) mx8[(e >> 1) & 7] = fmax3(mx8[(e >> 1) & 7], s[e], s[e + 1]);
      const float mt =
          fmax3(fmax3(mx8[0], mx8[1], mx8[2]), fmax3(mx8[3], mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])) * c;
      const bool need = mt > m_used + kRescaleThreshold;
      float alpha = 1.f;
      if (need) {
        alpha = fast_exp2(m_used - mt);  // m_used = -inf: 0
        l *= alpha;
        sg *= alpha;
        m_used = mt;
      }
      const float msub = m_used == -INFINITY ? 0.f : m_used;
      // Pairs of columns in packed fp32; one pair in four takes its
      // exponentials from the FMA-pipe polynomial, the rest from MUFU, which
      // balances the two units (MUFU alone was the softmax's bottleneck).
      const uint64_t c2 = f2(c, c), nm2 = f2(-msub, -msub);
      uint64_t lp[2] = {f2(0.f, 0.f), f2(0.f, 0.f)}, sp[2] = {f2(0.f, 0.f), f2(0.f, 0.f)};
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        // S is all in registers, so P may now overwrite it in TMEM.
        float t[32];
        tmem_ld32(cs + COL_T + 32 * hf, t);
        tmem_wait_ld();
        uint32_t pk[16], ptk[16];
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          const uint64_t x = ffma2(f2(s[32 * hf + e], s[32 * hf + e + 1]), c2, nm2);
          const uint64_t p = ((e >> 1) & 3) == 3 ? exp2_poly2(x)
                                                 : f2(fast_exp2(f2lo(x)), fast_exp2(f2hi(x)));
          const uint64_t pt = fmul2(p, f2(t[e], t[e + 1]));
          lp[(e >> 1) & 1] = fadd2(lp[(e >> 1) & 1], p);
          sp[(e >> 1) & 1] = fadd2(sp[(e >> 1) & 1], pt);
          pk[e >> 1] = pack_bf16x2(p);
          ptk[e >> 1] = pack_bf16x2(pt);
        }
        tmem_st16(cs + 16 * hf, pk);
        tmem_st16(cs + COL_T + 16 * hf, ptk);  // T[0,32) was read in half 0
      }
      const uint64_t lsum = fadd2(lp[0], lp[1]), ssum = fadd2(sp[0], sp[1]);
      l += f2lo(lsum) + f2hi(lsum);
      sg += f2lo(ssum) + f2hi(ssum);
      tmem_wait_st();
      if (j > 0) {
        // The previous tile's value UMMAs must be done before O is touched
        // and before P of this tile is handed over.
        ok = mbar_wait(smem_u32(&pv_done[(j - 1) & 1]), ((j - 1) >> 1) & 1, ab);
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
      ok = mbar_wait(smem_u32(&pv_done[(ntiles - 1) & 1]), ((ntiles - 1) >> 1) & 1, ab);
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
    if (warp == SM_WARP0 && lane == 0 && !ab.raised()) {
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
