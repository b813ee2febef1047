// Backward pass of the causal Parallax prefill on the tcgen05 tensor cores
// (bf16 operands, fp32 accumulation in TMEM, TMA loads), d = 128.
//
// The pages ("Parallax: parametrized local linear attention for language
// modeling", section "Core mechanism" for the forward, section
// "Experimental results" for the training runs) print no backward pass. With
// w the causal softmax weights of query i, t_j = rho_i . k_j,
// sbar = sum_j w_j t_j and c_j = 1 + sbar - t_j, the forward is
// o = sum_j w_j c_j v_j. For an output gradient g, with u_j = g . v_j,
// a = g . o^SA and D = g . o + a sbar, differentiating gives
//   dv_j   += w_j c_j g
//   dt_j    = w_j (a - u_j)
//   ds_j    = w_j (c_j u_j + a t_j - D)        (score gradient)
//   dq      = tau sum_j ds_j k_j,   drho = sum_j dt_j k_j
//   dk_j   += tau ds_j q + dt_j rho
// (the tests check this form against autograd through the explicit
// covariance). The forward saves lse, o^SA and sbar per row; a small kernel
// turns them into a record per row, {-lse log2 e, 1 + sbar, a, -D}, stored
// interleaved by pairs of rows ({x0, x1, y0, y1, ...}, 32 bytes per pair) so
// that two adjacent queries' records load as packed fp32x2 operands.
//
// Two kernels then stream the causal pairs, each with the same TMEM plan
// (512 columns): S [0,64) T [64,128) U [128,192) packed bf16 score and probe
// gradients [192,224) [224,256), two fp32 accumulators [256,384) [384,512).
//   bwd_dq_kernel: one CTA per 128 query rows; per 64-key tile
//     S = Q K^T, T = R K^T, U = dO V^T; dS, dT; dQ += dS K, dR += dT K.
//   bwd_dkv_kernel: one CTA per 128 keys of one kv head, over every query
//     head of its group and every 64-query tile at or after the keys;
//     [S^T | T^T] = K [Q; R]^T (one N = 128 product: S^T and T^T share the
//     A operand K, so stacking Q and R reads K once per K step) and
//     U^T = V dO^T; then dV += (w c)^T dO and dK += dS^T Q + dT^T R.
// Neither kernel needs atomics: each output row is owned by one CTA. The
// elementwise warps release S, T and U as soon as they have loaded them
// (stu_free), so the next tile's score UMMAs run under the elementwise work
// and the current tile's gradient UMMAs. The key-block kernel has 12 warps:
// 0 TMA producer; 1, 2, 3 one UMMA-issuing thread each (warp 1 also
// allocates TMEM); 4..11 elementwise (two warps per TMEM lane quarter, each
// taking half of the tile's 64 columns; there is no row reduction, so the
// columns split freely). The query-block kernel has a fourth issuing thread
// (warp 4) for its gradient products and elementwise warps 5..12. The UMMAs
// are spread over several threads because one thread cannot issue
// tcgen05.mma as fast as the tensor core retires these shapes (measured
// 50-100 cycles per issue under load against 48-64 cycles of work).
#include <math.h>

#include <type_traits>

#include "plx_device.cuh"
#include "plx_internal.h"

namespace plx {
namespace {

constexpr int D = 128;
constexpr int THREADS = 32 * 12;
constexpr int EW_WARP0 = 4;               // first elementwise warp
constexpr int NEW = 256;                  // elementwise threads
constexpr uint32_t COL_S = 0, COL_T = 64, COL_U = 128, COL_GS = 192, COL_GT = 224;
constexpr uint32_t COL_ACC0 = 256, COL_ACC1 = 384;
constexpr int STAT_ROWS = 64;             // stats rows are padded to this multiple

struct BwdArgs {
  __nv_bfloat16 *g0, *g1;  // dq, dr (dq kernel) or dv, dk (dkv kernel)
  const float *stats;      // [B * Hq][Lpad / 2][8] row-pair records (see above)
  int B, Hq, Hkv, L, Lpad;
  float scale_log2, tau;
  unsigned *err;
};

// ---------------------------------------------------------------- per-row records
// Half a warp per (padded) row, 16 bytes of each tensor per lane:
// a = g . o^SA, D = g . o + a sbar.
__device__ __forceinline__ float dot8(uint4 x, uint4 y) {
  const uint32_t xs[4] = {x.x, x.y, x.z, x.w}, ys[4] = {y.x, y.y, y.z, y.w};
  float acc = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&xs[i]));
    const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&ys[i]));
    acc = fmaf(a.x, b.x, fmaf(a.y, b.y, acc));
  }
  return acc;
}

__global__ void __launch_bounds__(256) bwd_prep_kernel(
    const __nv_bfloat16 *__restrict__ out, const __nv_bfloat16 *__restrict__ o1,
    const __nv_bfloat16 *__restrict__ dout, const float *__restrict__ lse,
    const float *__restrict__ sbar, float *__restrict__ stats, int L, int Lpad, long long nrows) {
  const long long p = static_cast<long long>(blockIdx.x) * 16 + (threadIdx.x >> 4);
  const int sub = threadIdx.x & 15;
  if (p >= nrows) return;  // uniform per half warp; nrows is even, so whole warps exit together
  const long long zh = p / Lpad;
  const int i = static_cast<int>(p - zh * Lpad);
  float *rec = stats + (p >> 1) * 8 + (p & 1);  // Lpad is even: pairs stay within a head
  float go = 0.f, ga = 0.f;
  const bool valid = i < L;
  const long long row = zh * L + i;
  if (valid) {
    const size_t off = static_cast<size_t>(row) * D + sub * 8;
    const uint4 gv = *reinterpret_cast<const uint4 *>(dout + off);
    go = dot8(gv, *reinterpret_cast<const uint4 *>(out + off));
    ga = dot8(gv, *reinterpret_cast<const uint4 *>(o1 + off));
  }
#pragma unroll
  for (int sh = 8; sh > 0; sh >>= 1) {
    go += __shfl_xor_sync(0xffffffffu, go, sh);
    ga += __shfl_xor_sync(0xffffffffu, ga, sh);
  }
  if (sub == 0) {
    if (valid) {
      const float sb = sbar[row];
      rec[0] = -lse[row] * 1.4426950408889634f;
      rec[2] = 1.f + sb;
      rec[4] = ga;
      rec[6] = -fmaf(ga, sb, go);
    } else {
      // Padding rows: weight 2^-inf = 0 for every key.
      rec[0] = -INFINITY;
      rec[2] = 1.f;
      rec[4] = 0.f;
      rec[6] = 0.f;
    }
  }
}

// Gradients of two adjacent (query, key) pairs in packed fp32x2 arithmetic.
// Inputs: raw scores s, probe products t, u = g . v for the two pairs, and
// per pair the record {lse log2 e, 1 + sbar, a, D} split into packed
// components (for the query-block kernel both pairs share one query, for the
// key-block kernel they are two queries). Outputs: tau ds and dt (and w c
// when PC) as packed bf16. MASK: the pair block reaches the causal diagonal
// and m0 / m1 drop the pairs whose key lies after the query.
struct Stat2 {
  uint64_t nlse, s1, a, nd;  // -lse log2 e, 1 + sbar, a, -D
};
struct Grad2 {
  uint32_t gs, gt, pc;
};
template <bool MASK, bool PC>
__device__ __forceinline__ Grad2 grad_pair(uint64_t s, uint64_t t, uint64_t u, const Stat2 &st,
                                           bool m0, bool m1, uint64_t c2, uint64_t tau2) {
  const uint64_t neg1 = f2(-1.f, -1.f);
  const uint64_t x = ffma2(s, c2, st.nlse);
  float w0 = fast_exp2(f2lo(x)), w1 = fast_exp2(f2hi(x));
  if (MASK) {
    w0 = m0 ? 0.f : w0;
    w1 = m1 ? 0.f : w1;
  }
  const uint64_t w = f2(w0, w1);
  const uint64_t cc = ffma2(t, neg1, st.s1);                // 1 + sbar - t
  const uint64_t dd = ffma2(cc, u, ffma2(st.a, t, st.nd));  // c u + a t - D
  Grad2 r;
  r.gs = pack_bf16x2(fmul2(fmul2(w, tau2), dd));
  r.gt = pack_bf16x2(fmul2(w, ffma2(u, neg1, st.a)));       // w (a - u)
  if (PC) r.pc = pack_bf16x2(fmul2(w, cc));
  return r;
}

// Reads 128 fp32 TMEM columns [col, col + 64) of this thread's lane as two
// 32-column pieces, converts to bf16 and stores them at dst (64 values).
__device__ __forceinline__ void store_acc_half(uint32_t taddr, __nv_bfloat16 *dst, bool valid) {
#pragma unroll 1
  for (int part = 0; part < 2; ++part) {
    float v[32];
    tmem_ld32(taddr + part * 32, v);
    tmem_wait_ld();
    if (valid) {
      uint32_t pk[16];
#pragma unroll
      for (int e = 0; e < 32; e += 2) pk[e >> 1] = pack_bf16x2(v[e], v[e + 1]);
      uint4 *d4 = reinterpret_cast<uint4 *>(dst + part * 32);
#pragma unroll
      for (int u = 0; u < 4; ++u) d4[u] = make_uint4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
    }
  }
}

// =================================================================== dQ, dR
namespace qk {
constexpr int BM = 128;                        // query rows per CTA
constexpr int BN = 64;                         // keys per tile
constexpr int NST = 3;                         // K / V ring stages
constexpr int HALF_Q = BM * 64 * 2;            // 16 KB
constexpr int HALF_KV = BN * 64 * 2;           // 8 KB
constexpr int TILE_KV = 2 * HALF_KV;
constexpr int OFF_Q = 0, OFF_R = 2 * HALF_Q, OFF_DO = 4 * HALF_Q;
constexpr int OFF_K = 6 * HALF_Q;              // 98304
constexpr int OFF_V = OFF_K + NST * TILE_KV;   // 147456
constexpr int OFF_BAR = OFF_V + NST * TILE_KV; // 196608
constexpr int NBAR = 1 + 4 * NST + 5 + 4;
constexpr int SMEM_BYTES = OFF_BAR + NBAR * 8 + 16 + 1024;
// 13 warps: 0 TMA producer; 1, 2, 3 issue S, T, U; 4 issues the gradient
// products dQ and dR; 5..12 elementwise. The gradient products get a thread
// of their own: a thread that issues the next tile's score products blocks
// while the tensor queue is full and would take up the gradient hand-over
// late.
constexpr int Q_THREADS = 32 * 13;
constexpr int Q_EW_WARP0 = 5;
}  // namespace qk

__global__ void __launch_bounds__(qk::Q_THREADS, 1)
    bwd_dq_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_r,
                  const __grid_constant__ CUtensorMap tm_do, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const BwdArgs a) {
  using namespace qk;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + OFF_BAR);
  uint64_t *q_full = bars;              // Q, R, dO loaded
  uint64_t *k_full = bars + 1;
  uint64_t *k_empty = k_full + NST;     // dQ and dR UMMAs of the tile done
  uint64_t *v_empty = k_empty + NST;    // U UMMAs of the tile done
  uint64_t *v_full = v_empty + NST;
  uint64_t *stu_full = v_full + NST;    // count 3: S, T, U of the tile in TMEM
  uint64_t *stu_free = stu_full + 1;    // count 8 (a lane per elementwise warp): S, T, U loaded
  uint64_t *gs_full = stu_free + 1;     // count 8: dS, dT written
  uint64_t *acc_done = gs_full + 1;     // dQ and dR UMMAs of the tile done
  uint64_t *acc_full = acc_done + 1;    // every gradient UMMA done (epilogue)
  uint64_t *drain = acc_full + 1;       // [4] one per issuing thread
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + NBAR);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nqt = (a.L + BM - 1) / BM, per = a.B * a.Hq;
  const int o = blockIdx.x;
  const int qt = nqt - 1 - o / per, rem = o % per;
  const int h = rem % a.Hq, b = rem / a.Hq;
  const int zq = b * a.Hq + h, zk = b * a.Hkv + h / (a.Hq / a.Hkv);
  const int q0 = qt * BM;
  const int n = (min(q0 + BM, a.L) + BN - 1) / BN;

  if (threadIdx.x == 0) {
    mbar_init(smem_u32(q_full), 1);
    for (int s = 0; s < NST; ++s) {
      mbar_init(smem_u32(&k_full[s]), 1);
      mbar_init(smem_u32(&k_empty[s]), 1);
      mbar_init(smem_u32(&v_full[s]), 1);
      mbar_init(smem_u32(&v_empty[s]), 1);
    }
    mbar_init(smem_u32(stu_full), 3);
    mbar_init(smem_u32(stu_free), NEW / 32);  // a lane per elementwise warp
    mbar_init(smem_u32(gs_full), NEW / 32);
    mbar_init(smem_u32(acc_done), 1);
    mbar_init(smem_u32(acc_full), 1);
    for (int x = 0; x < 4; ++x) mbar_init(smem_u32(&drain[x]), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tensormap(&tm_q);
    prefetch_tensormap(&tm_r);
    prefetch_tensormap(&tm_do);
    prefetch_tensormap(&tm_k);
    prefetch_tensormap(&tm_v);
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
      const bool in_bounds = PLX_IN_BOUNDS(q0 >= 0 && q0 < a.L && zq < a.B * a.Hq && zk < a.B * a.Hkv &&
                                               (n - 1) * BN < a.L,
                                           ab);
      if (in_bounds) mbar_arrive_expect_tx(qb, 6 * HALF_Q);
      if (in_bounds) {
      tma_load_3d(smem_u32(smem + OFF_Q), &tm_q, 0, q0, zq, qb);
      tma_load_3d(smem_u32(smem + OFF_Q + HALF_Q), &tm_q, 64, q0, zq, qb);
      tma_load_3d(smem_u32(smem + OFF_R), &tm_r, 0, q0, zq, qb);
      tma_load_3d(smem_u32(smem + OFF_R + HALF_Q), &tm_r, 64, q0, zq, qb);
      tma_load_3d(smem_u32(smem + OFF_DO), &tm_do, 0, q0, zq, qb);
      tma_load_3d(smem_u32(smem + OFF_DO + HALF_Q), &tm_do, 64, q0, zq, qb);
      }
      int k_issued = 0, v_issued = 0;
      for (int j = 0; in_bounds && j < n; ++j) {
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
        if (in_bounds) mbar_wait_drain(qb, 0);
        for (int j = max(0, k_issued - NST); j < k_issued; ++j)
          mbar_wait_drain(smem_u32(&k_full[j % NST]), (j / NST) & 1);
        for (int j = max(0, v_issued - NST); j < v_issued; ++j)
          mbar_wait_drain(smem_u32(&v_full[j % NST]), (j / NST) & 1);
      }
    }
  } else if (warp < Q_EW_WARP0) {
    if (lane == 0) {
      // ---------------------------------------------------------- UMMA issuers
      // role 0: S = Q K^T; role 1: T = R K^T; role 2: U = dO V^T (K-major
      // operands); role 3: dQ += dS K and dR += dT K (K MN-major).
      const int role = warp - 1;
      bool ok = mbar_wait(smem_u32(q_full), 0, ab);
      if (role < 3) {
        constexpr uint32_t idesc_s = idesc_bf16_f32(BM, BN, 0);
        const uint64_t adesc =
            smem_desc_sw128(smem_u32(smem + (role == 0 ? OFF_Q : role == 1 ? OFF_R : OFF_DO)), 16, 1024);
        const uint64_t bdesc0 = smem_desc_sw128(smem_u32(smem + (role == 2 ? OFF_V : OFF_K)), 16, 1024);
        const uint32_t dcol = tbase + (role == 0 ? COL_S : role == 1 ? COL_T : COL_U);
        uint64_t *b_full = role == 2 ? v_full : k_full;
        // The operand stage of tile j is normally loaded before S, T, U of
        // tile j - 1 are free: wait for it first, so that only that
        // hand-over stands before the issue.
        auto operand_ready = [&](int j) -> bool {
          return mbar_wait(smem_u32(&b_full[j % NST]), (j / NST) & 1, ab);
        };
        auto issue_score = [&](int j) {
          const int st = j % NST;
          tc_fence_after();
          const uint64_t bd = bdesc0 + st * (TILE_KV >> 4);
#pragma unroll
          for (int ks = 0; ks < D / 16; ++ks)
            umma_ss(dcol, adesc + (ks >> 2) * (HALF_Q >> 4) + (ks & 3) * 2,
                    bd + (ks >> 2) * (HALF_KV >> 4) + (ks & 3) * 2, idesc_s, ks > 0);
          umma_commit(smem_u32(stu_full));
          if (role == 2) umma_commit(smem_u32(&v_empty[st]));
        };
        if (ok && operand_ready(0)) issue_score(0);
        for (int j = 0; ok && j + 1 < n; ++j) {
          // S, T, U of tile j are in registers once stu_free completes.
          if (!operand_ready(j + 1) || !mbar_wait_spin(smem_u32(stu_free), j & 1, ab)) break;
          issue_score(j + 1);
        }
      } else {
        constexpr uint32_t idesc_g = idesc_bf16_f32(BM, D, 1);
        const uint64_t kmn0 = smem_desc_sw128(smem_u32(smem + OFF_K), HALF_KV, 1024);
        for (int j = 0; ok && j < n; ++j) {
          if (!mbar_wait_spin(smem_u32(gs_full), j & 1, ab)) break;
          tc_fence_after();
          const int st = j % NST;
          const uint64_t km = kmn0 + st * (TILE_KV >> 4);
#pragma unroll
          for (int ks = 0; ks < BN / 16; ++ks)
            umma_ts(tbase + COL_ACC0, tbase + COL_GS + ks * 8, km + ks * (2048 >> 4), idesc_g,
                    (j > 0 || ks > 0));
#pragma unroll
          for (int ks = 0; ks < BN / 16; ++ks)
            umma_ts(tbase + COL_ACC1, tbase + COL_GT + ks * 8, km + ks * (2048 >> 4), idesc_g,
                    (j > 0 || ks > 0));
          umma_commit(smem_u32(acc_done));
          umma_commit(smem_u32(&k_empty[st]));
        }
        umma_commit(smem_u32(acc_full));
      }
      umma_commit(smem_u32(&drain[role]));
      mbar_wait_drain(smem_u32(&drain[role]), 0);
    }
  } else {
    // ------------------------------------------------------------ elementwise
    const int qw = warp & 3, hf = (warp - Q_EW_WARP0) >> 2;
    const int row = qw * 32 + lane, grow = q0 + row;
    const uint32_t tl = tbase + (static_cast<uint32_t>(qw * 32) << 16);
    float nl = -INFINITY, s1 = 1.f, aa = 0.f, nd = 0.f;
    if (grow < a.L) {
      const float *rec = a.stats + ((static_cast<size_t>(zq) * a.Lpad + grow) >> 1) * 8 + (grow & 1);
      nl = rec[0];
      s1 = rec[2];
      aa = rec[4];
      nd = rec[6];
    }
    const Stat2 st2{f2(nl, nl), f2(s1, s1), f2(aa, aa), f2(nd, nd)};
    const uint64_t c2 = f2(a.scale_log2, a.scale_log2), tau2 = f2(a.tau, a.tau);
    bool ok = true;
    for (int j = 0; j < n; ++j) {
      ok = mbar_wait(smem_u32(stu_full), j & 1, ab);
      if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      tc_fence_after();
      float s[32], t[32], u[32];
      tmem_ld32(tl + COL_S + 32 * hf, s);
      tmem_ld32(tl + COL_T + 32 * hf, t);
      tmem_ld32(tl + COL_U + 32 * hf, u);
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(stu_free));
      const int kbase = j * BN + 32 * hf;
      uint32_t gs[16], gt[16];
      if (j * BN + BN - 1 > q0) {  // the tile reaches the diagonal
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          const Grad2 g2 = grad_pair<true, false>(f2(s[e], s[e + 1]), f2(t[e], t[e + 1]),
                                                  f2(u[e], u[e + 1]), st2, kbase + e > grow,
                                                  kbase + e + 1 > grow, c2, tau2);
          gs[e >> 1] = g2.gs;
          gt[e >> 1] = g2.gt;
        }
      } else {
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          const Grad2 g2 = grad_pair<false, false>(f2(s[e], s[e + 1]), f2(t[e], t[e + 1]),
                                                   f2(u[e], u[e + 1]), st2, false, false, c2, tau2);
          gs[e >> 1] = g2.gs;
          gt[e >> 1] = g2.gt;
        }
      }
      if (j > 0) {
        // The previous tile's dQ / dR UMMAs read the gradient columns.
        ok = mbar_wait(smem_u32(acc_done), (j - 1) & 1, ab);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        tc_fence_after();
      }
      tmem_st16(tl + COL_GS + 16 * hf, gs);
      tmem_st16(tl + COL_GT + 16 * hf, gt);
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(gs_full));
    }
    if (ok) {
      ok = mbar_wait(smem_u32(acc_full), 0, ab);
      if (__all_sync(0xffffffffu, ok)) {
        tc_fence_after();
        const bool valid = grow < a.L;
        const size_t ro = (static_cast<size_t>(zq) * a.L + (valid ? grow : 0)) * D + 64 * hf;
        store_acc_half(tl + COL_ACC0 + 64 * hf, a.g0 + ro, valid);
        store_acc_half(tl + COL_ACC1 + 64 * hf, a.g1 + ro, valid);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
}

// =================================================================== dK, dV
namespace kv {
constexpr int BM = 128;                        // keys per CTA
constexpr int BN = 64;                         // queries per step
constexpr int NST = 3;                         // Q / R / dO ring stages
constexpr int HALF_K = BM * 64 * 2;            // 16 KB
constexpr int HALF_Q = BN * 64 * 2;            // 8 KB
constexpr int TILE_Q = 2 * HALF_Q;             // 16 KB
// A stage holds the 64 queries' Q, R and dO as [Q h0 | R h0 | Q h1 | R h1 |
// dO h0 | dO h1] (h0, h1: dims 0-63 and 64-127): within each half Q's rows
// are followed by R's, so [Q; R] is one K-major operand of 128 rows and
// S^T and T^T come from one N = 128 product that reads K once.
constexpr int STAGE = 3 * TILE_Q;
constexpr int OFF_K = 0, OFF_V = 2 * HALF_K;
constexpr int OFF_P = 4 * HALF_K;              // 65536: (w c)^T tile, 128 keys x 64 queries bf16
constexpr int OFF_STG = OFF_P + BM * BN * 2;   // 81920
// The per-row records of a step's 64 queries (1 KB, 32 row pairs of 32 bytes)
// in a ring of their own, read by every elementwise lane as broadcasts.
constexpr int REC_STAGES = 2;
constexpr int REC_BYTES = BN * 16;
constexpr int OFF_REC = OFF_STG + NST * STAGE;  // 229376
constexpr int OFF_BAR = OFF_REC + REC_STAGES * REC_BYTES;
constexpr int NBAR = 1 + 2 * NST + 5 + 3 + 2 * REC_STAGES;
// No alignment slack: the dynamic shared memory starts 1024-byte aligned
// (checked at run time), which is what leaves room for the records.
constexpr int SMEM_BYTES = OFF_BAR + NBAR * 8 + 16;
static_assert(SMEM_BYTES <= 232448, "dK/dV kernel shared memory");
}  // namespace kv

__global__ void __launch_bounds__(THREADS, 1)
    bwd_dkv_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_r,
                   const __grid_constant__ CUtensorMap tm_do, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const BwdArgs a) {
  using namespace kv;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *smem = smem_raw;
  if ((smem_u32(smem_raw) & 1023u) != 0u) {
    // The swizzled tiles need a 1024-byte aligned base; never expected.
    if (threadIdx.x == 0 && a.err) atomicOr(a.err, kErrLayout);
    return;
  }
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + OFF_BAR);
  uint64_t *kv_full = bars;             // K and V blocks loaded
  uint64_t *q_full = bars + 1;          // [NST] Q, R, dO of a step loaded
  uint64_t *q_empty = q_full + NST;     // [NST] count 2: the step's dV and dK UMMAs done
  uint64_t *stu_full = q_empty + NST;   // count 3
  uint64_t *stu_free = stu_full + 1;    // count 8 (a lane per elementwise warp)
  uint64_t *gs_full = stu_free + 1;     // count 8: (w c)^T in smem, dS^T / dT^T in TMEM
  uint64_t *acc_done = gs_full + 1;     // count 2
  uint64_t *acc_full = acc_done + 1;    // count 2
  uint64_t *drain = acc_full + 1;       // [3]
  uint64_t *rec_full = drain + 3;       // [REC_STAGES] a step's records loaded
  uint64_t *rec_empty = rec_full + REC_STAGES;  // [REC_STAGES] count 8: read by every elementwise warp
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + NBAR);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int per = a.B * a.Hkv, G = a.Hq / a.Hkv;
  const int o = blockIdx.x;
  const int kb = o / per, rem = o % per;  // key blocks in ascending order: longest first
  const int kvh = rem % a.Hkv, b = rem / a.Hkv;
  const int zk = b * a.Hkv + kvh;
  const int k0 = kb * BM;
  const int qt_lo = k0 / BN, nqt = (a.L + BN - 1) / BN;
  const int per_head = nqt - qt_lo;
  const int n = G * per_head;             // steps: every query head of the group x query tiles

  if (threadIdx.x == 0) {
    mbar_init(smem_u32(kv_full), 1);
    for (int s = 0; s < NST; ++s) {
      mbar_init(smem_u32(&q_full[s]), 1);
      mbar_init(smem_u32(&q_empty[s]), 2);
    }
    mbar_init(smem_u32(stu_full), 2);  // [S^T | T^T] and U^T
    mbar_init(smem_u32(stu_free), NEW / 32);  // a lane per elementwise warp
    mbar_init(smem_u32(gs_full), NEW / 32);
    mbar_init(smem_u32(acc_done), 2);
    mbar_init(smem_u32(acc_full), 2);
    for (int x = 0; x < 3; ++x) mbar_init(smem_u32(&drain[x]), 1);
    for (int x = 0; x < REC_STAGES; ++x) {
      mbar_init(smem_u32(&rec_full[x]), 1);
      mbar_init(smem_u32(&rec_empty[x]), NEW / 32);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tensormap(&tm_q);
    prefetch_tensormap(&tm_r);
    prefetch_tensormap(&tm_do);
    prefetch_tensormap(&tm_k);
    prefetch_tensormap(&tm_v);
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
      const uint32_t kvb = smem_u32(kv_full);
      int rec_issued = 0;
      const bool in_bounds = PLX_IN_BOUNDS(k0 >= 0 && k0 < a.L && zk < a.B * a.Hkv &&
                                               (b * a.Hq + (kvh + 1) * G) <= a.B * a.Hq,
                                           ab);
      if (in_bounds) mbar_arrive_expect_tx(kvb, 4 * HALF_K);
      if (in_bounds) {
      tma_load_3d(smem_u32(smem + OFF_K), &tm_k, 0, k0, zk, kvb);
      tma_load_3d(smem_u32(smem + OFF_K + HALF_K), &tm_k, 64, k0, zk, kvb);
      tma_load_3d(smem_u32(smem + OFF_V), &tm_v, 0, k0, zk, kvb);
      tma_load_3d(smem_u32(smem + OFF_V + HALF_K), &tm_v, 64, k0, zk, kvb);
      }
      int issued = 0;
      for (int s = 0; in_bounds && s < n; ++s) {
        const int st = s % NST;
        if (s >= NST && !mbar_wait(smem_u32(&q_empty[st]), ((s / NST) - 1) & 1, ab)) break;
        const int zq = b * a.Hq + kvh * G + s / per_head, y = (qt_lo + s % per_head) * BN;
        if (!PLX_IN_BOUNDS(zq < a.B * a.Hq && y < a.L, ab)) break;
        const uint32_t qf = smem_u32(&q_full[st]);
        const uint32_t base = smem_u32(smem + OFF_STG + st * STAGE);
        mbar_arrive_expect_tx(qf, STAGE);
        tma_load_3d(base, &tm_q, 0, y, zq, qf);
        tma_load_3d(base + HALF_Q, &tm_r, 0, y, zq, qf);
        tma_load_3d(base + 2 * HALF_Q, &tm_q, 64, y, zq, qf);
        tma_load_3d(base + 3 * HALF_Q, &tm_r, 64, y, zq, qf);
        tma_load_3d(base + 2 * TILE_Q, &tm_do, 0, y, zq, qf);
        tma_load_3d(base + 2 * TILE_Q + HALF_Q, &tm_do, 64, y, zq, qf);
        issued = s + 1;
        // The step's 64 query records, contiguous in the record array.
        const int rs = s % REC_STAGES;
        if (s >= REC_STAGES && !mbar_wait(smem_u32(&rec_empty[rs]), ((s / REC_STAGES) - 1) & 1, ab)) break;
        if (!PLX_IN_BOUNDS(y + BN <= a.Lpad, ab)) break;
        const uint32_t rf = smem_u32(&rec_full[rs]);
        mbar_arrive_expect_tx(rf, REC_BYTES);
        bulk_g2s(smem_u32(smem + OFF_REC + rs * REC_BYTES),
                 a.stats + (static_cast<size_t>(zq) * a.Lpad + y) * 4, REC_BYTES, rf);
        rec_issued = s + 1;
      }
      if (ab.raised()) {
        if (in_bounds) mbar_wait_drain(kvb, 0);
        for (int s = max(0, issued - NST); s < issued; ++s)
          mbar_wait_drain(smem_u32(&q_full[s % NST]), (s / NST) & 1);
        for (int s = max(0, rec_issued - REC_STAGES); s < rec_issued; ++s)
          mbar_wait_drain(smem_u32(&rec_full[s % REC_STAGES]), (s / REC_STAGES) & 1);
      }
    }
  } else if (warp < EW_WARP0) {
    if (lane == 0) {
      // ---------------------------------------------------------- UMMA issuers
      // role 0: [S^T | T^T] = K [Q; R]^T (one N = 128 product; its columns
      // are S^T [0, 64) and T^T [64, 128)) and dV += (w c)^T dO; role 1:
      // dK += (tau dS)^T Q + dT^T R (one thread, so the accumulator's first
      // write comes first); role 2: U^T = V dO^T.
      const int role = warp - 1;
      const bool scores = role != 1;
      constexpr uint32_t idesc_st = idesc_bf16_f32(BM, 2 * BN, 0);
      constexpr uint32_t idesc_u = idesc_bf16_f32(BM, BN, 0);
      constexpr uint32_t idesc_g = idesc_bf16_f32(BM, D, 1);
      const uint64_t adesc = smem_desc_sw128(smem_u32(smem + (role == 2 ? OFF_V : OFF_K)), 16, 1024);
      const uint64_t pdesc = smem_desc_sw128(smem_u32(smem + OFF_P), 16, 1024);
      // The score operand in K-major view: [Q; R] (128 rows, dim halves
      // 2 HALF_Q apart) for role 0, dO (64 rows, halves HALF_Q apart) for
      // role 2. MN-major views for the gradients: Q and R (halves 2 HALF_Q
      // apart), dO (HALF_Q apart).
      const uint64_t stg_k = smem_desc_sw128(smem_u32(smem + OFF_STG + (role == 2 ? 2 * TILE_Q : 0)), 16, 1024);
      const uint32_t slab = role == 2 ? (HALF_Q >> 4) : (2 * HALF_Q >> 4);
      const uint64_t qr_mn = smem_desc_sw128(smem_u32(smem + OFF_STG), 2 * HALF_Q, 1024);
      const uint64_t do_mn = smem_desc_sw128(smem_u32(smem + OFF_STG + 2 * TILE_Q), HALF_Q, 1024);
      const uint32_t dcol = tbase + (role == 2 ? COL_U : COL_S);
      const uint32_t idesc_s = role == 2 ? idesc_u : idesc_st;
      bool ok = mbar_wait(smem_u32(kv_full), 0, ab);
      auto operand_ready = [&](int s) -> bool {
        return mbar_wait(smem_u32(&q_full[s % NST]), (s / NST) & 1, ab);
      };
      auto issue_score = [&](int s) -> bool {
        const int st = s % NST;
        tc_fence_after();
        const uint64_t bd = stg_k + st * (STAGE >> 4);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks)
          umma_ss(dcol, adesc + (ks >> 2) * (HALF_K >> 4) + (ks & 3) * 2,
                  bd + (ks >> 2) * slab + (ks & 3) * 2, idesc_s, ks > 0);
        umma_commit(smem_u32(stu_full));
        return true;
      };
      if (scores) ok = ok && operand_ready(0) && issue_score(0);
      for (int s = 0; ok && s < n; ++s) {
        if (scores && s + 1 < n) {
          if (!operand_ready(s + 1) || !mbar_wait_spin(smem_u32(stu_free), s & 1, ab) ||
              !issue_score(s + 1))
            break;
        }
        if (role == 2) continue;
        if (!mbar_wait_spin(smem_u32(gs_full), s & 1, ab)) break;
        const int st = s % NST;
        // The stage's loads completed before its score products ran (role 0
        // waited on q_full); role 1 observes that too before reading Q and R.
        if (!scores && !mbar_wait(smem_u32(&q_full[st]), (s / NST) & 1, ab)) break;
        tc_fence_after();
        const uint64_t qm = qr_mn + st * (STAGE >> 4);
        const uint64_t rm = qm + (HALF_Q >> 4), om = do_mn + st * (STAGE >> 4);
        if (role == 0) {
#pragma unroll
          for (int ks = 0; ks < BN / 16; ++ks)
            umma_ss(tbase + COL_ACC0, pdesc + ks * 2, om + ks * (2048 >> 4), idesc_g, (s > 0 || ks > 0));
        } else {
#pragma unroll
          for (int ks = 0; ks < BN / 16; ++ks)
            umma_ts(tbase + COL_ACC1, tbase + COL_GS + ks * 8, qm + ks * (2048 >> 4), idesc_g, (s > 0 || ks > 0));
#pragma unroll
          for (int ks = 0; ks < BN / 16; ++ks)
            umma_ts(tbase + COL_ACC1, tbase + COL_GT + ks * 8, rm + ks * (2048 >> 4), idesc_g, 1);
        }
        umma_commit(smem_u32(acc_done));
        umma_commit(smem_u32(&q_empty[st]));
      }
      if (role != 2) umma_commit(smem_u32(acc_full));
      umma_commit(smem_u32(&drain[role]));
      mbar_wait_drain(smem_u32(&drain[role]), 0);
    }
  } else {
    // ------------------------------------------------------------ elementwise
    const int qw = warp & 3, hf = (warp - EW_WARP0) >> 2;
    const int row = qw * 32 + lane, krow = k0 + row;
    const uint32_t tl = tbase + (static_cast<uint32_t>(qw * 32) << 16);
    // This thread's row of the (w c)^T tile: 128-byte rows, 16-byte chunks
    // XOR-swizzled by the row index within each 8-row group (SW128, K-major).
    uint8_t *prow = smem + OFF_P + (row >> 3) * 1024 + (row & 7) * 128;
    const uint64_t c2 = f2(a.scale_log2, a.scale_log2), tau2 = f2(a.tau, a.tau);
    bool ok = true;
    for (int s = 0; s < n; ++s) {
      const int qbase = (qt_lo + s % per_head) * BN + 32 * hf;
      // The records of this half's 32 queries: 16 row pairs of two float4,
      // {-lse log2 e, 1 + sbar} and {a, -D} of both rows, read from the
      // step's record stage as broadcasts (every lane the same address).
      const int rs = s % REC_STAGES;
      const float4 *rec4 =
          reinterpret_cast<const float4 *>(smem + OFF_REC + rs * REC_BYTES) + 32 * hf;
      ok = mbar_wait(smem_u32(&rec_full[rs]), (s / REC_STAGES) & 1, ab);
      ok = ok && mbar_wait(smem_u32(stu_full), s & 1, ab);
      if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      tc_fence_after();
      float sv[32], tv[32], uv[32];
      tmem_ld32(tl + COL_S + 32 * hf, sv);
      tmem_ld32(tl + COL_T + 32 * hf, tv);
      tmem_ld32(tl + COL_U + 32 * hf, uv);
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(stu_free));
      uint32_t gs[16], gt[16], pc[16];
      auto cols = [&](auto mask_tag) {
        constexpr bool M = decltype(mask_tag)::value;
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          // Pair (qbase + e, qbase + e + 1): float4s e and e + 1 of the half.
          const float4 r0 = rec4[e], r1 = rec4[e + 1];
          const Stat2 st2{f2(r0.x, r0.y), f2(r0.z, r0.w), f2(r1.x, r1.y), f2(r1.z, r1.w)};
          const Grad2 g2 = grad_pair<M, true>(f2(sv[e], sv[e + 1]), f2(tv[e], tv[e + 1]),
                                              f2(uv[e], uv[e + 1]), st2, krow > qbase + e,
                                              krow > qbase + e + 1, c2, tau2);
          gs[e >> 1] = g2.gs;
          gt[e >> 1] = g2.gt;
          pc[e >> 1] = g2.pc;
        }
      };
      // Mask only where the block reaches the causal diagonal.
      if (k0 + BM - 1 > (qt_lo + s % per_head) * BN) cols(std::true_type{});
      else cols(std::false_type{});
      // The records are read: their stage may be reloaded.
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&rec_empty[rs]));
      if (s > 0) {
        ok = mbar_wait(smem_u32(acc_done), (s - 1) & 1, ab);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        tc_fence_after();
      }
#pragma unroll
      for (int ch = 0; ch < 4; ++ch) {
        const int cidx = 4 * hf + ch;
        *reinterpret_cast<uint4 *>(prow + ((cidx ^ (row & 7)) << 4)) =
            make_uint4(pc[4 * ch], pc[4 * ch + 1], pc[4 * ch + 2], pc[4 * ch + 3]);
      }
      tmem_st16(tl + COL_GS + 16 * hf, gs);
      tmem_st16(tl + COL_GT + 16 * hf, gt);
      tmem_wait_st();
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(gs_full));
    }
    if (ok) {
      ok = mbar_wait(smem_u32(acc_full), 0, ab);
      if (__all_sync(0xffffffffu, ok)) {
        tc_fence_after();
        const bool valid = krow < a.L;
        const size_t ro = (static_cast<size_t>(zk) * a.L + (valid ? krow : 0)) * D + 64 * hf;
        store_acc_half(tl + COL_ACC0 + 64 * hf, a.g0 + ro, valid);
        store_acc_half(tl + COL_ACC1 + 64 * hf, a.g1 + ro, valid);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
}

}  // namespace

size_t prefill_bwd_stats_count(int B, int Hq, int L) {
  const size_t lpad = (static_cast<size_t>(L) + STAT_ROWS - 1) / STAT_ROWS * STAT_ROWS;
  return static_cast<size_t>(B) * Hq * lpad;
}

cudaError_t launch_prefill_bwd(const void *q, const void *k, const void *v, const void *r,
                               const void *out, const void *o1, const float *lse,
                               const float *sbar, const void *dout, void *dq, void *dk, void *dv,
                               void *dr, int B, int Hq, int Hkv, int L, void *stats, unsigned *err,
                               cudaStream_t stream) {
  static thread_local unsigned long long configured_ctx = 0;
  const unsigned long long ctx = context_id();
  if (ctx == 0 || configured_ctx != ctx) {
    cudaError_t e = cudaFuncSetAttribute(bwd_dq_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         qk::SMEM_BYTES);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(bwd_dkv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               kv::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    configured_ctx = ctx;
  }
  EncodeTiledFn enc = encode_tiled_fn();
  if (enc == nullptr) return cudaErrorInvalidValue;
  const int Lpad = (L + STAT_ROWS - 1) / STAT_ROWS * STAT_ROWS;
  float *st = static_cast<float *>(stats);
  const long long nrows = static_cast<long long>(B) * Hq * Lpad;
  bwd_prep_kernel<<<static_cast<unsigned>((nrows + 15) / 16), 256, 0, stream>>>(
      static_cast<const __nv_bfloat16 *>(out), static_cast<const __nv_bfloat16 *>(o1),
      static_cast<const __nv_bfloat16 *>(dout), lse, sbar, st, L, Lpad, nrows);

  BwdArgs a;
  a.stats = st;
  a.B = B;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.L = L;
  a.Lpad = Lpad;
  a.scale_log2 = 1.4426950408889634f / sqrtf(static_cast<float>(D));
  a.tau = 1.f / sqrtf(static_cast<float>(D));
  a.err = err;

  CUtensorMap mq, mr, mo, mk, mv;
  // dQ / dR: 128-row query boxes, 64-row key boxes.
  if (!make_head_rows_map(enc, &mq, q, L, B * Hq, qk::BM) ||
      !make_head_rows_map(enc, &mr, r, L, B * Hq, qk::BM) ||
      !make_head_rows_map(enc, &mo, dout, L, B * Hq, qk::BM) ||
      !make_head_rows_map(enc, &mk, k, L, B * Hkv, qk::BN) ||
      !make_head_rows_map(enc, &mv, v, L, B * Hkv, qk::BN))
    return cudaErrorInvalidValue;
  a.g0 = static_cast<__nv_bfloat16 *>(dq);
  a.g1 = static_cast<__nv_bfloat16 *>(dr);
  const int nq = (L + qk::BM - 1) / qk::BM * B * Hq;
  bwd_dq_kernel<<<nq, qk::Q_THREADS, qk::SMEM_BYTES, stream>>>(mq, mr, mo, mk, mv, a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;

  // dK / dV: 64-row query boxes, 128-row key boxes.
  if (!make_head_rows_map(enc, &mq, q, L, B * Hq, kv::BN) ||
      !make_head_rows_map(enc, &mr, r, L, B * Hq, kv::BN) ||
      !make_head_rows_map(enc, &mo, dout, L, B * Hq, kv::BN) ||
      !make_head_rows_map(enc, &mk, k, L, B * Hkv, kv::BM) ||
      !make_head_rows_map(enc, &mv, v, L, B * Hkv, kv::BM))
    return cudaErrorInvalidValue;
  a.g0 = static_cast<__nv_bfloat16 *>(dv);
  a.g1 = static_cast<__nv_bfloat16 *>(dk);
  const int nk = (L + kv::BM - 1) / kv::BM * B * Hkv;
  bwd_dkv_kernel<<<nk, THREADS, kv::SMEM_BYTES, stream>>>(mq, mr, mo, mk, mv, a);
  return cudaGetLastError();
}

}  // namespace plx
