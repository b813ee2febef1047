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
// Chunked prefill: the L queries may be the last L positions of Lk >= L keys
// (a new chunk against an existing cache); query row i then sees keys
// 0 .. Lk - L + i. Plain prefill is Lk = L.
//
// Persistent: one CTA per SM walks a list of work items (128 query rows of
// one (batch, head)), longest first, dealt to the CTAs in snake order so the
// causal work evens out. TMEM, barriers and the pipelines stay up across
// items, and barrier phases follow CTA-wide tile and item counters. A
// dedicated epilogue warpgroup writes an item's output while the softmax
// warps already work on the next item; the next item's first value UMMAs
// wait for the epilogue to have read O (o_free). 13 warps:
//   warp 0      TMA producer: Q and R per item (128 x 128 each, loaded as
//               soon as the previous item's last S/T UMMAs finish), then K_j
//               and V_j (64 keys x 128 each) into two 4-stage rings, 128-byte
//               swizzled. A K stage is freed once the S and T UMMAs that read
//               it finish, a V stage once the value UMMAs finish.
//   warp 1      TMEM allocator; one thread issues O1 += P V.
//   warp 2      one thread issues O2 += (P o T) V.
//   warps 3..6  softmax: thread = query row = TMEM lane.
//   warps 7, 8  one thread each issues S = Q K^T and T = R K^T.
//   warps 9..12 epilogue: reads O1, O2 and the softmax's row statistics,
//               writes o and lse.
// Four issuing threads, because one thread cannot issue tcgen05.mma as fast
// as the tensor core retires these shapes (measured: 50-100 cycles per issue
// under load against 48-64 cycles of work per instruction). The value
// UMMAs, which sit on the critical path (softmax -> P V -> next softmax), have
// issuers of their own that respond at once. S and T of tile j + 2 overwrite
// P(j) and P o T(j), so they must execute after the value UMMAs of tile j:
// each value issuer signals pv_issued once its UMMAs are issued (after a
// tcgen05 before-thread-sync fence), and the score issuer waits for that
// signal (then an after-thread-sync fence) and issues behind them. The
// tensor pipe executes UMMAs in that order, so the score UMMAs queue right
// behind the value UMMAs instead of waiting for them to complete.
// Tensor memory (512 columns x 128 lanes, fp32):
//   [0,64) S_0  [64,128) T_0  [128,192) S_1  [192,256) T_1  (double buffered)
//   [256,384) O1              [384,512) O2
// The softmax writes P and P o T as packed bf16 (S_x[0,32) = P, T_x[0,32) =
// P o T) and the value GEMMs read them straight from TMEM (A-from-TMEM
// form), V from shared memory (MN-major). P is handed over in two halves of
// 32 keys, so the first two K steps of the value UMMAs start while the
// softmax still works on the second half; an O rescale (rare with the lazy
// max) happens before either half is handed over. Rescaling is lazy: the max used in
// the exponent only moves when a row's tile max exceeds it by more than
// 2^8, which keeps every quantity exact (they all share the stale max) and
// rarely touches O in TMEM.
#include <math.h>

#include <type_traits>

#include "plx_device.cuh"
#include "plx_internal.h"

namespace plx {
namespace {

constexpr int D = 128;
constexpr int BM = 128;                       // query rows per work item
constexpr int BN = 64;                        // keys per tile
constexpr int NST = 4;                        // stages per K / V ring
constexpr int HALF_Q = BM * 64 * 2;           // 16 KB: 128 rows x 64 dims
constexpr int HALF_KV = BN * 64 * 2;          // 8 KB: 64 rows x 64 dims
constexpr int TILE_KV = 2 * HALF_KV;          // 16 KB: one K or V tile
constexpr int OFF_Q = 0;
constexpr int OFF_R = 2 * HALF_Q;
constexpr int OFF_K = 4 * HALF_Q;             // 65536
constexpr int OFF_V = OFF_K + NST * TILE_KV;  // 131072
constexpr int OFF_STAT = OFF_V + NST * TILE_KV;  // 196608: [2][3][BM] row statistics
// Output staging: per epilogue warp two 2 KB boxes (o and o^SA) of 32 rows x
// 32 dims bf16, 64-byte rows with the 64-byte swizzle of the store map.
constexpr int OFF_OST = OFF_STAT + 2 * 3 * BM * 4;  // 199680, a multiple of 1024
constexpr int OST_BOX = 32 * 32 * 2;
constexpr int OFF_BAR = OFF_OST + 4 * 2 * OST_BOX;
constexpr int NBAR = 2 + 4 * NST + 2 + 4 + 2 + 4 + 1 + 2 + 4;
constexpr int SMEM_BYTES = OFF_BAR + NBAR * 8 + 16 + 1024;  // + alignment slack
constexpr int SM_WARP0 = 3;                   // first softmax warp
constexpr int EP_WARP0 = 9;                   // first epilogue warp
constexpr int THREADS = 32 * 13;
constexpr uint32_t COL_S0 = 0, COL_S1 = 128, COL_T = 64, COL_O1 = 256, COL_O2 = 384;
constexpr float kRescaleThreshold = 8.0f;     // log2 units

struct PrefillArgs {
  __nv_bfloat16 *out;
  float *lse;
  float *cor;  // optional: |correction| / |o| per row
  __nv_bfloat16 *o1;  // optional (training): o^SA = O1 / l per row, bf16
  float *sbar;        // optional (training): sigma / l per row
  int Hq, Hkv, L, B, nqt, nitems;
  int Lk, qoff;  // keys per head; absolute position of query row 0 (Lk - L)
  float scale_log2;  // log2(e) / sqrt(d)
  unsigned *err;
};

struct Item {
  int q0, ntiles, zq, zk;
};

// k-th work item of this CTA: rounds of gridDim.x items, longest first,
// dealt left-to-right in even rounds and right-to-left in odd ones. All CTAs
// work on the same round at about the same time, so the K/V tiles the round's
// items stream stay in L2 between the CTAs that read them.
__device__ __forceinline__ bool item_of(const PrefillArgs &a, int k, Item &it) {
  const int G = gridDim.x;
  const int pos = (k & 1) ? G - 1 - static_cast<int>(blockIdx.x) : static_cast<int>(blockIdx.x);
  const int o = k * G + pos;
  if (o >= a.nitems) return false;
  const int per_qt = a.Hq * a.B;
  const int qt = a.nqt - 1 - o / per_qt;
  const int rem = o % per_qt;
  const int h = rem % a.Hq, b = rem / a.Hq;
  it.q0 = qt * BM;
  it.ntiles = (min(a.qoff + it.q0 + BM, a.Lk) + BN - 1) / BN;
  it.zq = b * a.Hq + h;
  it.zk = b * a.Hkv + h / (a.Hq / a.Hkv);
  return true;
}

__global__ void __launch_bounds__(THREADS, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_r,
                      const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                      const __grid_constant__ CUtensorMap tm_o, const __grid_constant__ CUtensorMap tm_o1,
                      const PrefillArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
  float *stat = reinterpret_cast<float *>(smem + OFF_STAT);  // [item parity][m, l, sigma][row]
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + OFF_BAR);
  uint64_t *q_full = bars;             // Q and R of the item loaded
  uint64_t *q_empty = bars + 1;        // the item's last S and T UMMAs done (count 2)
  uint64_t *k_full = bars + 2;
  uint64_t *k_empty = k_full + NST;    // count 2 (S and T)
  uint64_t *v_full = k_empty + NST;
  uint64_t *v_empty = v_full + NST;    // count 2 (O1 and O2)
  uint64_t *st_full = v_empty + NST;   // [2] count 2
  uint64_t *p_full = st_full + 2;      // [2][2] count 4 (a lane per softmax warp): P of keys [32 h, 32 h + 32) of buffer x
  uint64_t *pv_done = p_full + 4;      // [2] count 2: value UMMAs of the tiles in buffer x
  uint64_t *pv_issued = pv_done + 2;   // [2][2]: O1 (h = 0) / O2 (h = 1) value UMMAs of buffer x issued
  uint64_t *o_free = pv_issued + 4;      // count 4 (a lane per epilogue warp): the epilogue has read O1 and O2
  uint64_t *stat_full = o_free + 1;    // [2] count 4: row statistics of an item written
  uint64_t *drain = stat_full + 2;     // [4]: one per issuing thread
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + NBAR);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(smem_u32(q_full), 1);
    mbar_init(smem_u32(q_empty), 2);
    for (int s = 0; s < NST; ++s) {
      mbar_init(smem_u32(&k_full[s]), 1);
      mbar_init(smem_u32(&k_empty[s]), 2);
      mbar_init(smem_u32(&v_full[s]), 1);
      mbar_init(smem_u32(&v_empty[s]), 2);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(smem_u32(&st_full[x]), 2);
      mbar_init(smem_u32(&p_full[2 * x]), 4);
      mbar_init(smem_u32(&p_full[2 * x + 1]), 4);
      mbar_init(smem_u32(&pv_done[x]), 2);
      mbar_init(smem_u32(&pv_issued[2 * x]), 1);
      mbar_init(smem_u32(&pv_issued[2 * x + 1]), 1);
      mbar_init(smem_u32(&stat_full[x]), 4);
    }
    mbar_init(smem_u32(o_free), 4);
    for (int x = 0; x < 4; ++x) mbar_init(smem_u32(&drain[x]), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tensormap(&tm_q);
    prefetch_tensormap(&tm_r);
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
      int g = 0, k_issued = 0, v_issued = 0, q_issued = 0;
      bool ok = true;
      Item it;
      for (int k = 0; ok && item_of(a, k, it); ++k) {
        // Q and R of the previous item are dead once its last S/T UMMAs finish.
        if (k > 0 && !mbar_wait(smem_u32(q_empty), (k - 1) & 1, ab)) break;
        // Every box of the item lies inside its head's rows (TMA zero-fills
        // past L or Lk only within a head).
        if (!PLX_IN_BOUNDS(it.q0 >= 0 && it.q0 < a.L && it.zq >= 0 && it.zq < a.B * a.Hq &&
                               it.zk >= 0 && it.zk < a.B * a.Hkv && it.ntiles >= 1 &&
                               (it.ntiles - 1) * BN < a.Lk,
                           ab))
          break;
        mbar_arrive_expect_tx(qb, 4 * HALF_Q);
        tma_load_3d(smem_u32(smem + OFF_Q), &tm_q, 0, it.q0, it.zq, qb);
        tma_load_3d(smem_u32(smem + OFF_Q + HALF_Q), &tm_q, 64, it.q0, it.zq, qb);
        tma_load_3d(smem_u32(smem + OFF_R), &tm_r, 0, it.q0, it.zq, qb);
        tma_load_3d(smem_u32(smem + OFF_R + HALF_Q), &tm_r, 64, it.q0, it.zq, qb);
        q_issued = k + 1;
        for (int j = 0; j < it.ntiles; ++j) {
          const int gg = g + j, st = gg % NST;
          if (gg >= NST && !mbar_wait(smem_u32(&k_empty[st]), ((gg / NST) - 1) & 1, ab)) { ok = false; break; }
          const uint32_t kf = smem_u32(&k_full[st]);
          mbar_arrive_expect_tx(kf, TILE_KV);
          const uint32_t kb = smem_u32(smem + OFF_K + st * TILE_KV);
          tma_load_3d(kb, &tm_k, 0, j * BN, it.zk, kf);
          tma_load_3d(kb + HALF_KV, &tm_k, 64, j * BN, it.zk, kf);
          k_issued = gg + 1;
          if (gg >= NST && !mbar_wait(smem_u32(&v_empty[st]), ((gg / NST) - 1) & 1, ab)) { ok = false; break; }
          const uint32_t vf = smem_u32(&v_full[st]);
          mbar_arrive_expect_tx(vf, TILE_KV);
          const uint32_t vb = smem_u32(smem + OFF_V + st * TILE_KV);
          tma_load_3d(vb, &tm_v, 0, j * BN, it.zk, vf);
          tma_load_3d(vb + HALF_KV, &tm_v, 64, j * BN, it.zk, vf);
          v_issued = gg + 1;
        }
        g += it.ntiles;
      }
      if (ab.raised()) {
        // Let this thread's own copies land before the CTA exits.
        if (q_issued > 0) mbar_wait_drain(qb, (q_issued - 1) & 1);
        for (int gg = max(0, k_issued - NST); gg < k_issued; ++gg)
          mbar_wait_drain(smem_u32(&k_full[gg % NST]), (gg / NST) & 1);
        for (int gg = max(0, v_issued - NST); gg < v_issued; ++gg)
          mbar_wait_drain(smem_u32(&v_full[gg % NST]), (gg / NST) & 1);
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
      int g = 0;
      bool ok = true;
      Item it;
      for (int k = 0; ok && item_of(a, k, it); ++k) {
        for (int j = 0; j < it.ntiles; ++j) {
          const int gg = g + j, x = gg & 1, st = gg % NST;
          // V and O are normally ready long before P: waiting on them first
          // leaves only the P hand-over between the softmax and the issue.
          // The first value UMMA of an item overwrites O: the previous item's
          // epilogue must have read it.
          if (j == 0 && k > 0 && !mbar_wait_spin(smem_u32(o_free), (k - 1) & 1, ab)) { ok = false; break; }
          if (!mbar_wait(smem_u32(&v_full[st]), (gg / NST) & 1, ab)) { ok = false; break; }
          if (!mbar_wait_spin(smem_u32(&p_full[2 * x]), (gg >> 1) & 1, ab)) { ok = false; break; }
          tc_fence_after();
          const uint64_t vdesc = vdesc0 + st * (TILE_KV >> 4);
          const uint32_t ap = tbase + (x ? COL_S1 : COL_S0) + col_off;
#pragma unroll
          for (int ks = 0; ks < BN / 16; ++ks) {
            if (ks == 2 && !mbar_wait_spin(smem_u32(&p_full[2 * x + 1]), (gg >> 1) & 1, ab)) { ok = false; break; }
            umma_ts(dout, ap + ks * 8, vdesc + ks * (2048 >> 4), idesc_pv, (j > 0 || ks > 0));
          }
          if (!ok) break;
          umma_commit(smem_u32(&pv_done[x]));
          umma_commit(smem_u32(&v_empty[st]));
          // The score UMMAs of tile gg + 2 may now be issued behind these.
          tc_fence_before();
          mbar_arrive(smem_u32(&pv_issued[2 * x + (is_o1 ? 0 : 1)]));
        }
        g += it.ntiles;
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
      int g = 0;
      bool ok = true;
      Item it;
      for (int k = 0; ok && item_of(a, k, it); ++k) {
        if (!mbar_wait(smem_u32(q_full), k & 1, ab)) break;
        for (int j = 0; j < it.ntiles; ++j) {
          const int gg = g + j, x = gg & 1, st = gg % NST;
          // K is normally loaded well ahead: wait for it first. Buffer x holds
          // P (P o T) of CTA tile gg - 2: its value UMMAs must have been
          // issued; issued earlier, they execute first.
          if (!mbar_wait(smem_u32(&k_full[st]), (gg / NST) & 1, ab)) { ok = false; break; }
          if (gg >= 2 && !mbar_wait_spin(smem_u32(&pv_issued[2 * x + (is_s ? 0 : 1)]), ((gg - 2) >> 1) & 1, ab)) { ok = false; break; }
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
        if (ok) umma_commit(smem_u32(q_empty));  // Q / R of this item no longer read
        g += it.ntiles;
      }
      umma_commit(smem_u32(&drain[is_s ? 2 : 3]));
      mbar_wait_drain(smem_u32(&drain[is_s ? 2 : 3]), 0);
    }
  } else if (warp >= SM_WARP0 && warp < SM_WARP0 + 4) {
    // ------------------------------------------------------------ softmax
    const int qw = warp & 3;             // TMEM lane quarter this warp may touch
    const int row = qw * 32 + lane;      // query row within the item
    const uint32_t tl = tbase + (static_cast<uint32_t>(qw * 32) << 16);
    const float c = a.scale_log2;
    int g = 0;
    bool ok = true;
    Item it;
    for (int k = 0; ok && item_of(a, k, it); ++k) {
      const int n = it.ntiles, q0 = it.q0, grow = q0 + row;
      float m_used = -INFINITY, l = 0.f, sg = 0.f;
      for (int j = 0; j < n; ++j) {
        const int gg = g + j, x = gg & 1;
        ok = mbar_wait(smem_u32(&st_full[x]), (gg >> 1) & 1, ab);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        tc_fence_after();
        const uint32_t cs = tl + (x ? COL_S1 : COL_S0);
        float s[64];
        tmem_ld32(cs, *reinterpret_cast<float(*)[32]>(&s[0]));
        tmem_ld32(cs + 32, *reinterpret_cast<float(*)[32]>(&s[32]));
        tmem_wait_ld();
        if (j * BN + BN - 1 > a.qoff + q0) {  // tile reaches the diagonal: causal mask
#pragma unroll
          for (int e = 0; e < BN; ++e)
            if (j * BN + e > a.qoff + grow) s[e] = -INFINITY;
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
        if (j > 0 && __any_sync(0xffffffffu, need)) {
          // Rescaling O: the previous tile's value UMMAs must be done first.
          // Without a rescale P is handed over as soon as it is written; the
          // value UMMAs of one accumulator run in issue order, so tile j's
          // follow tile j-1's.
          ok = mbar_wait(smem_u32(&pv_done[(gg - 1) & 1]), ((gg - 1) >> 1) & 1, ab);
          if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
          tc_fence_after();
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
        const float msub = m_used == -INFINITY ? 0.f : m_used;
        // Pairs of columns in packed fp32; exponentials from MUFU (ex2).
        const uint64_t c2 = f2(c, c), nm2 = f2(-msub, -msub);
        uint64_t lp[2] = {f2(0.f, 0.f), f2(0.f, 0.f)}, sp[2] = {f2(0.f, 0.f), f2(0.f, 0.f)};
#pragma unroll
        for (int qq = 0; qq < 4; ++qq) {
          // Quarter qq reads T columns [16 qq, 16 qq + 16) and stores P over S
          // columns [8 qq, 8 qq + 8) (S is all in registers) and P o T over T
          // columns [8 qq, 8 qq + 8), which earlier quarters have read. T
          // comes in 16-column pieces: 13 warps leave 128 registers a thread.
          float t[16];
          tmem_ld16(cs + COL_T + 16 * qq, t);
          tmem_wait_ld();
          uint32_t pk[8], ptk[8];
#pragma unroll
          for (int e = 0; e < 16; e += 2) {
            const int col = 16 * qq + e;
            const uint64_t xx = ffma2(f2(s[col], s[col + 1]), c2, nm2);
            const uint64_t p = f2(fast_exp2(f2lo(xx)), fast_exp2(f2hi(xx)));
            const uint64_t pt = fmul2(p, f2(t[e], t[e + 1]));
            lp[(e >> 1) & 1] = fadd2(lp[(e >> 1) & 1], p);
            sp[(e >> 1) & 1] = fadd2(sp[(e >> 1) & 1], pt);
            pk[e >> 1] = pack_bf16x2(p);
            ptk[e >> 1] = pack_bf16x2(pt);
          }
          tmem_st8(cs + 8 * qq, pk);
          tmem_st8(cs + COL_T + 8 * qq, ptk);
          if (qq == 1) {
            // P of keys [0, 32) is in place: its value UMMAs may start.
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&p_full[2 * x]));
          }
        }
        const uint64_t lsum = fadd2(lp[0], lp[1]), ssum = fadd2(sp[0], sp[1]);
        l += f2lo(lsum) + f2hi(lsum);
        sg += f2lo(ssum) + f2hi(ssum);
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&p_full[2 * x + 1]));
      }
      if (!ok) break;
      // Hand the row statistics to the epilogue and move on to the next item.
      float *st = stat + (k & 1) * 3 * BM;
      st[row] = m_used;
      st[BM + row] = l;
      st[2 * BM + row] = sg;
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&stat_full[k & 1]));
      g += n;
    }
  } else if (warp >= EP_WARP0 && warp < EP_WARP0 + 4) {
    // ------------------------------------------------------------ epilogue
    // Each warp owns 32 rows. Per 32-dim part it writes its 32 x 32 box of o
    // (and of o^SA when asked) into its staging boxes and one lane stores
    // them with TMA: whole lines to global memory instead of 16-byte pieces
    // of 32 rows, which kept the warp's stores, and so the release of O,
    // waiting on the memory pipeline.
    const int qw = warp & 3;
    const int row = qw * 32 + lane;
    const uint32_t tl = tbase + (static_cast<uint32_t>(qw * 32) << 16);
    const uint32_t box_o = smem_u32(smem + OFF_OST + qw * 2 * OST_BOX), box_o1 = box_o + OST_BOX;
    // Row `lane` of a box: 64 bytes, 16-byte chunk c at c ^ ((lane >> 1) & 3).
    const uint32_t rbase = lane * 64, rsw = (lane >> 1) & 3;
    int g = 0;
    Item it;
    for (int k = 0; item_of(a, k, it); ++k) {
      const int glast = g + it.ntiles - 1, grow = it.q0 + row;
      g += it.ntiles;
      bool ok = mbar_wait(smem_u32(&stat_full[k & 1]), (k >> 1) & 1, ab);
      ok = ok && mbar_wait(smem_u32(&pv_done[glast & 1]), (glast >> 1) & 1, ab);
      if (!__all_sync(0xffffffffu, ok)) break;
      tc_fence_after();
      const float *st = stat + (k & 1) * 3 * BM;
      const float m_used = st[row], l = st[BM + row], sg = st[2 * BM + row];
      const float inv = 1.f / l;
      const float g1 = (1.f + sg * inv) * inv;
      // Correction (Sigma rho) = O2/l - (O1/l)(sigma/l); o = O1/l - correction.
      const float gc = sg * inv * inv;
      const bool want_cor = a.cor != nullptr, want_o1 = a.o1 != nullptr;
      const bool row_ok = grow < a.L &&
                          PLX_IN_BOUNDS(it.zq >= 0 && it.zq < a.B * a.Hq && grow >= 0, ab);
      // The warp's box holds rows q0 + 32 qw ..; the store map drops rows >= L.
      const bool box_live = it.q0 + qw * 32 < a.L;
      float csq = 0.f, osq = 0.f;
      // The optional outputs are compile-time choices of the part loop, so
      // its unrolled element loop carries no branch.
      auto drain = [&](auto cor_tag, auto o1_tag) {
        constexpr bool COR = decltype(cor_tag)::value, O1 = decltype(o1_tag)::value;
#pragma unroll 1
        for (int part = 0; part < 4; ++part) {
          float o1[32], o2[32];
          tmem_ld32(tl + COL_O1 + part * 32, o1);
          tmem_ld32(tl + COL_O2 + part * 32, o2);
          tmem_wait_ld();
          if (part == 3) {
            // O has been read: the next item's value UMMAs may overwrite it.
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(o_free));
          }
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            const float x0 = fmaf(o1[e], g1, -o2[e] * inv), x1 = fmaf(o1[e + 1], g1, -o2[e + 1] * inv);
            pk[e >> 1] = pack_bf16x2(x0, x1);
            if (COR) {
              const float c0 = fmaf(-o1[e], gc, o2[e] * inv), c1 = fmaf(-o1[e + 1], gc, o2[e + 1] * inv);
              csq = fmaf(c0, c0, fmaf(c1, c1, csq));
              osq = fmaf(x0, x0, fmaf(x1, x1, osq));
            }
          }
          if (box_live) {
            // The previous part's stores have read the staging boxes.
            if (lane == 0) bulk_wait_read_all();
            __syncwarp();
#pragma unroll
            for (int c = 0; c < 4; ++c)
              st_shared_v4(box_o + rbase + ((c ^ rsw) << 4), pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
            if (O1) {
              // Saved for the backward pass: o^SA = O1 / l.
#pragma unroll
              for (int e = 0; e < 32; e += 2) pk[e >> 1] = pack_bf16x2(o1[e] * inv, o1[e + 1] * inv);
#pragma unroll
              for (int c = 0; c < 4; ++c)
                st_shared_v4(box_o1 + rbase + ((c ^ rsw) << 4), pk[4 * c], pk[4 * c + 1], pk[4 * c + 2],
                             pk[4 * c + 3]);
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_store_3d(&tm_o, box_o, part * 32, it.q0 + qw * 32, it.zq);
              if (O1) tma_store_3d(&tm_o1, box_o1, part * 32, it.q0 + qw * 32, it.zq);
              bulk_commit_group();
            }
          }
        }
      };
      if (want_cor && want_o1) drain(std::true_type{}, std::true_type{});
      else if (want_cor) drain(std::true_type{}, std::false_type{});
      else if (want_o1) drain(std::false_type{}, std::true_type{});
      else drain(std::false_type{}, std::false_type{});
      if (a.lse != nullptr && row_ok)
        a.lse[static_cast<size_t>(it.zq) * a.L + grow] = (m_used + log2f(l)) * 0.6931471805599453f;
      if (a.sbar != nullptr && row_ok) a.sbar[static_cast<size_t>(it.zq) * a.L + grow] = sg * inv;
      if (want_cor && row_ok)
        a.cor[static_cast<size_t>(it.zq) * a.L + grow] = osq > 0.f ? sqrtf(csq) / sqrtf(osq) : 0.f;
    }
    // The staging boxes stay in use until the last stores have completed.
    if (lane == 0) bulk_wait_all();
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
}

}  // namespace

// Store map of a [heads][L][128] bf16 output: 32 x 32 boxes, 64-byte swizzle.
static bool make_out_store_map(EncodeTiledFn enc, CUtensorMap *map, const void *ptr, int L, int heads) {
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(L),
                              static_cast<cuuint64_t>(heads)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2,
                                 static_cast<cuuint64_t>(L) * D * 2};
  const cuuint32_t box[3] = {32, 32, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(ptr), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
             CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_head_rows_map(EncodeTiledFn enc, CUtensorMap *map, const void *ptr, int L, int heads,
                        int box_rows) {
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

cudaError_t launch_prefill_tc(const void *q, const void *k, const void *v, const void *r, void *out,
                              float *lse, float *cor, void *o1, float *sbar, int B, int Hq, int Hkv,
                              int L, int Lk, unsigned *err, cudaStream_t stream) {
  static thread_local unsigned long long configured_ctx = 0;
  const unsigned long long ctx = context_id();
  if (ctx == 0 || configured_ctx != ctx) {
    cudaError_t e = cudaFuncSetAttribute(prefill_tc_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) return e;
    configured_ctx = ctx;
  }
  EncodeTiledFn enc = encode_tiled_fn();
  if (enc == nullptr) return cudaErrorInvalidValue;
  CUtensorMap mq, mr, mk, mv, mo, mo1;
  if (!make_head_rows_map(enc, &mq, q, L, B * Hq, BM) || !make_head_rows_map(enc, &mr, r, L, B * Hq, BM) ||
      !make_head_rows_map(enc, &mk, k, Lk, B * Hkv, BN) || !make_head_rows_map(enc, &mv, v, Lk, B * Hkv, BN) ||
      !make_out_store_map(enc, &mo, out, L, B * Hq) ||
      !make_out_store_map(enc, &mo1, o1 != nullptr ? o1 : out, L, B * Hq))
    return cudaErrorInvalidValue;
  PrefillArgs a;
  a.out = static_cast<__nv_bfloat16 *>(out);
  a.lse = lse;
  a.cor = cor;
  a.o1 = static_cast<__nv_bfloat16 *>(o1);
  a.sbar = sbar;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.L = L;
  a.Lk = Lk;
  a.qoff = Lk - L;
  a.B = B;
  a.nqt = (L + BM - 1) / BM;
  a.nitems = a.nqt * Hq * B;
  a.scale_log2 = 1.4426950408889634f / sqrtf(static_cast<float>(D));
  a.err = err;
  const int grid = min(a.nitems, sm_count());
  prefill_tc_kernel<<<grid, THREADS, SMEM_BYTES, stream>>>(mq, mr, mk, mv, mo, mo1, a);
  return cudaGetLastError();
}

}  // namespace plx
