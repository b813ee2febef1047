// Parallax decode: equal shares of the batch's key stream streamed from a
// packed bf16 KV cache, then a log-sum-exp combine of the partial results.
//
// The method ("Parallax: parametrized local linear attention for language
// modeling", sections "Core mechanism" and "Hardware-aware algorithm") adds a
// covariance branch to softmax attention that reads the same KV stream; the
// pages' decode kernel therefore computes q.k and rho.k in the same tensor-core
// instructions so the cache is read from HBM once for both branches. This
// kernel does the same on sm_103a with warp-level mma.sync:
//
//   One wave of CTAs (two per SM), each with an equal share of the keys of
//   all (sequence, kv head) rows taken as one stream; a share is cut at row
//   boundaries into items. 4 consumer warps + 1 producer warp per CTA.
//   Producer: one thread issues tiled TMA loads of 16-token x 64-dim boxes of
//     the K and V cache (3-D tensor maps over [tokens, Hkv, d]) into a ring of
//     8 shared-memory stages, 128-byte swizzled so ldmatrix is bank-conflict
//     free; completion is counted in bytes on per-stage mbarriers. Four 2 KB
//     requests move an 8 KB stage (per-row 256-byte copies were limited by
//     the TMA request rate). The ring runs on across items.
//   Consumers: stages are dealt round-robin to the 4 warps, two per warp. For each 16 keys
//     one m16n8k16 product gives all four dot-product families at once: A rows
//     0..G-1 hold the G query heads' q, rows 8..8+G-1 their probes r, so the
//     accumulator row g is the score s = q.k and row g + 8 is t = r.k for the
//     same key in the same thread. P and P*T then form the A operand of the
//     value product (rows g: P -> O1, rows g + 8: P*T -> O2), again in
//     registers, with V^T read by ldmatrix.trans.
//   Each warp runs the online-softmax recurrence (running max m, denominator
//   l, sigma = sum p t, O1 and O2 accumulators, all rescaled together); at
//   the end of an item the warps are merged in shared memory and the CTA
//   writes one partial record per query head: (O1/l, O2/l, sigma/l,
//   log2-sum-exp) in fp32.
//
// The combine kernel merges the records of a (sequence, head) with weights
// 2^(lse_s - max) and only then forms o = O1 - O2 + O1 * s. Combining final
// per-share outputs would be wrong: O1 * s is bilinear in the partial sums.
#include <math.h>

#include <mutex>

#include "plx_device.cuh"
#include "plx_internal.h"

namespace plx {
namespace {

constexpr int D = 128;
constexpr int KT = 16;                        // keys per stage (one TMA box row count)
constexpr int NCW = 4;                        // consumer warps
constexpr int GMAX = 8;                       // query heads per kv head (A rows 0..7 and 8..15)
// Tile t goes to warp t % NCW and stage t % NST. NST is a multiple of NCW, so
// a stage is only ever consumed by one warp, which has itself consumed the
// stage's previous phase before it waits on the next one: a parity wait can
// never be two phases ahead (which it could not tell apart).
constexpr int NST = 2 * NCW;                  // stages in the ring
constexpr int HALF = KT * 128;                // one 64-dim half of KT rows, 128-byte swizzled
constexpr int STAGE_BYTES = 4 * HALF;         // K half 0, K half 1, V half 0, V half 1
constexpr int OFF_RED = NST * STAGE_BYTES;    // 65536: per-warp partials of one item
constexpr int RED_FLOATS = NCW * 2 * GMAX * D;
constexpr int OFF_MLS = OFF_RED + RED_FLOATS * 4;
constexpr int MLS_FLOATS = NCW * GMAX * 3;
constexpr int OFF_BAR = OFF_MLS + MLS_FLOATS * 4;
constexpr int OFF_FLAG = OFF_BAR + 2 * NST * 8;
constexpr int OFF_PLAN = OFF_FLAG + 16;
static_assert(NST % NCW == 0, "each stage must belong to one consumer warp");
static_assert(OFF_BAR % 8 == 0 && OFF_PLAN % 16 == 0, "barrier and plan alignment");
constexpr int SMEM_BYTES = OFF_PLAN + 64 + 1024;  // + alignment slack
constexpr int REC = 2 * D + 2;                // floats per partial record
constexpr int THREADS = 32 * (NCW + 1);
// The default schedule takes floor(sqrt(W)) CTAs for W keys (at most the
// grid): a small call's time is a fixed cost plus its longest share's
// stream, and on GB300 the fastest CTA counts (L2 flushed before each call)
// were 64 for 4096 keys (14.7 us against 20.7 with 8 CTAs of 512 keys), 128
// for 16384 (16.7 against 22.5) and 192 to 256 for 65536 (22.5 against 23.6
// with 128). For a batch of one length (whose shares are then aligned with
// the rows) at most kUniformMaxShares: from there on 256 CTAs beat the full
// grid of 304 by 1-6% (B = 2 x 8192: 24.8 against 26.2 us); a ragged batch ran
// 0.9% faster on the full grid.
constexpr long long kUniformMaxShares = 256;

struct DecodeArgs {
  const __nv_bfloat16 *q, *r;
  const int *seqlens;
  float *recs;  // [(nshare * G + B * Hq)][REC] partial records
  int2 *meta;   // [B * Hkv] {first record slot, number of slots} of each (sequence, kv head)
  int B, Hq, Hkv, G, nshare;
  bool dflt;         // default schedule: floor(sqrt(W)) shares; for a uniform batch at most 256, aligned with the rows
  float scale_log2;  // log2(e) / sqrt(d)
  unsigned *err;
};

// The CTA's share of the batch, worked out once by the producer warp.
struct Plan {
  long long W;      // keys of the whole batch over all kv heads
  long long s, e;   // this CTA's share [s, e) of the flattened key stream
  long long pb0;    // first token of sequence b0
  int n;            // CTAs with work (n <= gridDim.x)
  int b0;           // the sequence holding position s; -1: no work
};

// Byte offset of 16-byte chunk c (0..15 over the 128 dims) of row `row` in a
// stage half pair laid out by TMA with the 128-byte swizzle.
__device__ __forceinline__ uint32_t swz(int row, int c) {
  return (c >> 3) * HALF + row * 128 + ((((c & 7) ^ (row & 7))) << 4);
}

__device__ __forceinline__ void consumer_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(NCW * 32) : "memory");
}

// The batch is one flattened stream of keys: sequence b's kv head h holds the
// positions [Hkv P_b + h len_b, Hkv P_b + (h + 1) len_b), P_b the tokens in
// front of sequence b. CTA c of n takes [floor(c W / n), floor((c + 1) W / n))
// and cuts it at the (sequence, kv head) boundaries into items. Every warp
// walks the same items from the plan, so they agree on every item without
// talking to each other.
struct Item {
  int b, kvh, k0, k1;  // keys [k0, k1) of kv head kvh of sequence b
  int len;             // keys of sequence b
  long long tok0;      // first token of sequence b in the cache
};

struct Walk {
  long long pos, e, pb, row_base;
  int b, len;
  __device__ __forceinline__ Walk(const Plan &p, const int *seqlens, int Hkv)
      : pos(p.s), e(p.e), pb(p.pb0), row_base(p.pb0 * Hkv), b(p.b0),
        len(max(seqlens[p.b0], 0)) {}
  __device__ __forceinline__ bool next(Item &it, const int *seqlens, int Hkv) {
    if (pos >= e) return false;
    // Positions below W all lie in some sequence, so b stays below B here.
    while (pos >= row_base + static_cast<long long>(Hkv) * len) {
      pb += len;
      row_base = pb * Hkv;
      len = max(seqlens[++b], 0);
    }
    const long long off = pos - row_base;
    it.b = b;
    it.kvh = static_cast<int>(off / len);
    it.k0 = static_cast<int>(off - static_cast<long long>(it.kvh) * len);
    it.k1 = static_cast<int>(min(static_cast<long long>(len), it.k0 + (e - pos)));
    it.len = len;
    it.tok0 = pb;
    pos += it.k1 - it.k0;
    return true;
  }
};

__global__ void __launch_bounds__(THREADS)
    decode_split_kernel(const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_v, const DecodeArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + OFF_BAR);
  uint64_t *empty = full + NST;
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + OFF_FLAG);
  Plan *plan = reinterpret_cast<Plan *>(smem + OFF_PLAN);
  const int c = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (warp == NCW) {
    // ------------------------------------------------------------ plan
    long long T = 0;
    int nz = 0, lmin = 0x7fffffff, lmax = 0;  // over the sequences of nonzero length
#pragma unroll 4
    for (int i = lane; i < a.B; i += 32) {
      const int len = max(a.seqlens[i], 0);
      T += len;
      if (len > 0) {
        ++nz;
        lmin = min(lmin, len);
        lmax = max(lmax, len);
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      T += __shfl_xor_sync(0xffffffffu, T, o);
      nz += __shfl_xor_sync(0xffffffffu, nz, o);
      lmin = min(lmin, __shfl_xor_sync(0xffffffffu, lmin, o));
      lmax = max(lmax, __shfl_xor_sync(0xffffffffu, lmax, o));
    }
    if (T >= (1LL << 30)) {  // past the tensor maps' token extent: no work
      if (lane == 0 && c == 0 && a.err) atomicOr(a.err, kErrBadInput);
      T = 0;
      nz = 0;
    }
    const long long W = T * a.Hkv;
    long long n = W;
    if (a.dflt) {
      n = static_cast<long long>(sqrtf(static_cast<float>(W)));
      while (n > 0 && n * n > W) --n;
      while ((n + 1) * (n + 1) <= W) ++n;
      if (nz > 0 && lmin == lmax) n = min(n, kUniformMaxShares);
    }
    n = max(1LL, min(static_cast<long long>(a.nshare), n));
    if (a.dflt && nz > 0 && lmin == lmax) {
      // Rows of one length: cut every row at the same keys (k shares a row)
      // or give every share whole rows (m rows a share), so that the CTAs
      // streaming the kv heads of a sequence read the same tokens at the
      // same time (neighbouring 256-byte rows of the cache). Measured on
      // GB300 (B = 64, 8192 tokens): 256 aligned shares 6.58 TB/s, 304
      // unaligned 6.34. Taken only if it keeps 80% of the CTAs.
      const long long R = static_cast<long long>(nz) * a.Hkv, floor_n = (4 * n + 4) / 5;
      long long best = 0;
      if (R <= n) {
        best = R * (n / R);
      } else {
        for (long long m = (R + n - 1) / n, m_end = m + 64; m < m_end && R / m >= floor_n; ++m)
          if (R % m == 0) {
            best = R / m;
            break;
          }
      }
      if (best >= floor_n) n = best;
    }
    const long long s = c * W / n, e = (c + 1) * W / n;
    int b0 = -1;
    long long pb0 = 0;
    if (c < n && s < e) {
      // The first sequence whose flattened end lies past s.
      long long base = 0;
      for (int i0 = 0; i0 < a.B; i0 += 32) {
        const int i = i0 + lane;
        const long long len = i < a.B ? max(a.seqlens[i], 0) : 0;
        long long inc = len;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const long long v = __shfl_up_sync(0xffffffffu, inc, o);
          if (lane >= o) inc += v;
        }
        const unsigned hit = __ballot_sync(0xffffffffu, i < a.B && (base + inc) * a.Hkv > s);
        if (hit != 0u) {
          const int l = __ffs(hit) - 1;
          b0 = i0 + l;
          pb0 = base + __shfl_sync(0xffffffffu, inc - len, l);
          break;
        }
        base += __shfl_sync(0xffffffffu, inc, 31);
      }
    }
    if (lane == 0) {
      plan->W = W;
      plan->s = s;
      plan->e = e;
      plan->pb0 = pb0;
      plan->n = static_cast<int>(n);
      plan->b0 = b0;
    }
  }
  if (threadIdx.x == 0) {
    for (int st = 0; st < NST; ++st) {
      mbar_init(smem_u32(&full[st]), 1);
      mbar_init(smem_u32(&empty[st]), 1);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  // The combine kernel is launched as a programmatic dependent of this grid:
  // its blocks may be scheduled once every CTA here has passed this point,
  // and they wait (griddepcontrol.wait) for this grid to complete before
  // reading a record, so their launch overlaps this grid's tail.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const Plan pl = *plan;
  if (pl.b0 < 0) return;  // no share: more CTAs than the batch needs
  const Abort ab{abort_flag, a.err};

  // Tile t of an item covers keys [k0 + KT t, min(k0 + KT (t + 1), k1)). Its
  // TMA box of KT tokens starts at token min(tok0 + k0 + KT t, tok0 + k1 - KT),
  // so the box never reaches past the item's last key (and so never past the
  // cache); rows in front of the tile's first key (`skip` of them: keys of the
  // previous tile, of another sequence, or zero fill before token 0) are
  // masked by the consumer. Tiles are numbered across the CTA's items (g), so
  // stages and parities run on from one item to the next.
  if (warp == NCW) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tensormap(&tm_k);
      prefetch_tensormap(&tm_v);
      Walk wk(pl, a.seqlens, a.Hkv);
      Item it;
      int g = 0;
      bool ok = true;
      while (ok && wk.next(it, a.seqlens, a.Hkv)) {
        const int first = static_cast<int>(it.tok0) + it.k0, last = static_cast<int>(it.tok0) + it.k1;
        const int nt = (it.k1 - it.k0 + KT - 1) / KT;
        for (int t = 0; t < nt; ++t, ++g) {
          const int st = g % NST;
          if (g >= NST && !mbar_wait(smem_u32(&empty[st]), ((g / NST) - 1) & 1, ab)) {
            ok = false;
            break;
          }
          const int z = min(first + KT * t, last - KT);
          // The box stays inside the item's tokens (or, for a cache shorter
          // than one box, starts before token 0, where TMA zero-fills).
          if (!PLX_IN_BOUNDS(it.b < a.B && it.kvh < a.Hkv && z + KT <= last &&
                                 static_cast<long long>(last) * a.Hkv <= pl.W &&
                                 (z >= 0 || last < KT),
                             ab)) {
            ok = false;
            break;
          }
          const uint32_t bar = smem_u32(&full[st]);
          mbar_arrive_expect_tx(bar, STAGE_BYTES);
          const uint32_t base = smem_u32(smem + st * STAGE_BYTES);
          tma_load_3d(base, &tm_k, 0, it.kvh, z, bar);
          tma_load_3d(base + HALF, &tm_k, 64, it.kvh, z, bar);
          tma_load_3d(base + 2 * HALF, &tm_v, 0, it.kvh, z, bar);
          tma_load_3d(base + 3 * HALF, &tm_v, 64, it.kvh, z, bar);
        }
      }
      if (!ok) {
        // Let this thread's own copies (tiles g - NST .. g - 1) land before the CTA exits.
        for (int t = max(0, g - NST); t < g; ++t)
          mbar_wait_drain(smem_u32(&full[t % NST]), (t / NST) & 1);
      }
    }
    return;
  }

  // ------------------------------------------------------------ consumers
  // Every consumer warp takes part in every item's merge (both barriers),
  // also after an abort, so the named barrier is always complete.
  const int g = lane >> 2, tq = lane & 3;
  float *red = reinterpret_cast<float *>(smem + OFF_RED);  // [NCW][2G][D]
  float *mls = reinterpret_cast<float *>(smem + OFF_MLS);  // [NCW][G][3]
  Walk wk(pl, a.seqlens, a.Hkv);
  Item it;
  int gt = 0;  // tiles of the previous items
  while (wk.next(it, a.seqlens, a.Hkv)) {
    const int nt = (it.k1 - it.k0 + KT - 1) / KT;
    float acc[16][4];
    float m = -INFINITY, l = 0.f, sg = 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
    uint32_t qa[8][4];
    // The item's query rows and record slots lie inside q, r and the records.
    const bool item_ok = PLX_IN_BOUNDS(
        it.b < a.B && it.kvh < a.Hkv &&
            static_cast<long long>(it.b) * a.Hq + static_cast<long long>(it.kvh + 1) * a.G <=
                static_cast<long long>(a.B) * a.Hq &&
            c + it.b * a.Hkv + it.kvh < pl.n + a.B * a.Hkv,
        ab);
    {
      const bool live = g < a.G && item_ok;
      const size_t hrow = (static_cast<size_t>(it.b) * a.Hq + it.kvh * a.G + (live ? g : 0)) * D;
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
    for (int t = (warp - gt % NCW + NCW) % NCW; t < nt; t += NCW) {
      const int gi = gt + t;
      const int st = gi % NST;
      bool ok = false;
      if (lane == 0) ok = !ab.raised() && mbar_wait(smem_u32(&full[st]), (gi / NST) & 1, ab);
      if (!__shfl_sync(0xffffffffu, ok, 0)) continue;  // aborting: skip the tile
      const uint32_t kb = smem_u32(smem + st * STAGE_BYTES);
      const uint32_t vb = kb + 2 * HALF;
      // Rows [0, skip) of the box precede this tile's first key.
      const int skip = (it.k0 + KT * t) - min(it.k0 + KT * t, it.k1 - KT);
#pragma unroll
      for (int half = 0; half < KT / 16; ++half) {
        if (half * 16 + 15 < skip) continue;
        float cc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
        const int krow = half * 16 + (lane >> 4) * 8 + (lane & 7);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          uint32_t b0, b1, b2, b3;
          ldsm_x4(kb + swz(krow, 2 * kk + ((lane >> 3) & 1)), b0, b1, b2, b3);
          mma_bf16_16816(cc[0], qa[kk], b0, b1);
          mma_bf16_16816(cc[1], qa[kk], b2, b3);
        }
        // cc[n][0..1]: s for box rows half*16 + 8n + 2tq + {0,1}; cc[n][2..3]: t for the same rows.
        float s[2][2];
        float mx = -INFINITY;
#pragma unroll
        for (int n = 0; n < 2; ++n)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int row = half * 16 + 8 * n + 2 * tq + e;
            s[n][e] = row >= skip ? cc[n][e] * a.scale_log2 : -INFINITY;
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
            pt[n][e] = p[n][e] * cc[n][2 + e];
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
    gt += nt;
    l += __shfl_xor_sync(0xffffffffu, l, 1);
    l += __shfl_xor_sync(0xffffffffu, l, 2);
    sg += __shfl_xor_sync(0xffffffffu, sg, 1);
    sg += __shfl_xor_sync(0xffffffffu, sg, 2);

    // ---------------------------------------------------------- merge warps
    if (g < a.G) {
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
    consumer_sync();
    const int row = it.b * a.Hkv + it.kvh;
    const int dim = threadIdx.x;
    const bool aborted = ab.raised();
    for (int gh = 0; gh < a.G; ++gh) {
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < NCW; ++w) M = fmaxf(M, mls[(w * a.G + gh) * 3]);
      if (!item_ok) continue;
      float *rec = a.recs + (static_cast<size_t>(c + row) * a.G + gh) * REC;
      if (M == -INFINITY || aborted) {
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
    if (it.k0 == 0 && dim == 0 && item_ok) {
      // This CTA holds the row's first key, so it is the first of the CTAs
      // that hold the row (CTA c' writes its records to slot c' + row); the
      // last one holds the row's last key x, CTA floor(((x + 1) n - 1) / W).
      const long long x_last = (it.tok0 * a.Hkv + static_cast<long long>(it.kvh) * it.len) +
                               it.len - 1;
      const int c_last = static_cast<int>(((x_last + 1) * pl.n - 1) / pl.W);
      a.meta[row] = make_int2(c + row, c_last - c + 1);
    }
    consumer_sync();  // the next item's partials overwrite red and mls
  }
}

// One block of D threads per (sequence, query head): merge the row's records.
// They are read in parallel: each thread takes a strided share of the records'
// log-sum-exps for the maximum and the weights (staged in shared memory, CCH
// records at a time), then every thread accumulates its own dimension over
// the staged records with independent loads in flight.
constexpr int CCH = 512;

__device__ __forceinline__ float block_max(float v, float *slot) {
#pragma unroll
  for (int sh = 16; sh > 0; sh >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, sh));
  if ((threadIdx.x & 31) == 0) slot[threadIdx.x >> 5] = v;
  __syncthreads();
  v = slot[0];
#pragma unroll
  for (int w = 1; w < D / 32; ++w) v = fmaxf(v, slot[w]);
  return v;
}

__global__ void __launch_bounds__(D) decode_combine_kernel(const float *__restrict__ recs,
                                                          const int2 *__restrict__ meta,
                                                          const int *__restrict__ seqlens,
                                                          __nv_bfloat16 *__restrict__ out,
                                                          float *__restrict__ cor, int Hq,
                                                          int Hkv, int nslots) {
  __shared__ float wsig[2][CCH];
  __shared__ float slot[D / 32];
  // Launched as a programmatic dependent of the split kernel: wait for that
  // grid to complete (its records and row table visible) before any read.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int bh = blockIdx.x, dim = threadIdx.x;
  const int b = bh / Hq, h = bh - b * Hq, G = Hq / Hkv;
  const int kvh = h / G, gh = h - kvh * G;
  float o = 0.f, c = 0.f;
  if (seqlens[b] > 0) {  // a row of length 0 has no records: its output is 0
    const int2 mt = meta[b * Hkv + kvh];
    // Every row of nonzero length has its table entry written by this call's
    // split kernel; an entry outside the records (left by an earlier call
    // when this one did no work) is not followed.
    const bool inside = mt.x >= 0 && mt.y >= 1 && static_cast<long long>(mt.x) + mt.y <= nslots;
    const int nrec = inside ? mt.y : 0;
    const size_t stride = static_cast<size_t>(G) * REC;
    const float *rec =
        recs + static_cast<size_t>(inside ? mt.x : 0) * stride + static_cast<size_t>(gh) * REC;
    float M = -INFINITY;
    for (int s = dim; s < nrec; s += D) M = fmaxf(M, rec[s * stride + 2 * D + 1]);
    M = block_max(M, slot);  // the same value in every thread
    if (M != -INFINITY) {
      float W = 0.f, o1 = 0.f, o2 = 0.f, sf = 0.f;
      for (int base = 0; base < nrec; base += CCH) {
        const int cnt = min(CCH, nrec - base);
        const float *rb = rec + static_cast<size_t>(base) * stride;
        __syncthreads();  // the previous chunk's weights are consumed
        for (int i = dim; i < cnt; i += D) {
          const float w = exp2f(rb[i * stride + 2 * D + 1] - M);  // aborted share: lse = -inf, w = 0
          wsig[0][i] = w;
          wsig[1][i] = w * rb[i * stride + 2 * D];
        }
        __syncthreads();
#pragma unroll 8
        for (int i = 0; i < cnt; ++i) {
          const float w = wsig[0][i];
          W += w;
          sf += wsig[1][i];
          o1 = fmaf(w, rb[i * stride + dim], o1);
          o2 = fmaf(w, rb[i * stride + D + dim], o2);
        }
      }
      const float inv = 1.f / W;
      o1 *= inv;
      o2 *= inv;
      sf *= inv;
      c = o2 - o1 * sf;  // the correction Sigma rho
      o = o1 - c;
    }
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
                          int nshare, bool default_share, void *workspace, unsigned *err,
                          cudaStream_t stream) {
  static thread_local unsigned long long configured_ctx = 0;
  const unsigned long long ctx = context_id();
  if (ctx == 0 || configured_ctx != ctx) {
    cudaError_t e = cudaFuncSetAttribute(decode_split_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) return e;
    configured_ctx = ctx;
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
  a.meta = static_cast<int2 *>(workspace);
  a.recs = reinterpret_cast<float *>(static_cast<uint8_t *>(workspace) + decode_meta_bytes(B, Hkv));
  a.B = B;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.G = Hq / Hkv;
  a.nshare = nshare;
  a.dflt = default_share;
  a.scale_log2 = 1.4426950408889634f / sqrtf(static_cast<float>(D));
  a.err = err;
  decode_split_kernel<<<nshare, THREADS, SMEM_BYTES, stream>>>(mk, mv, a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(B * Hq);
  cfg.blockDim = dim3(D);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, decode_combine_kernel, static_cast<const float *>(a.recs),
                         static_cast<const int2 *>(a.meta), seqlens,
                         static_cast<__nv_bfloat16 *>(out), cor, Hq, Hkv, nshare + B * Hkv);
  if (e != cudaSuccess) return e;
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
// The array's address per device and the id of the context it was looked up
// in; a device reset destroys that context (and the array with it), and the
// next call looks the address up again in the new context.
float *g_noalloc_ptr[64] = {};
unsigned long long g_noalloc_ctx[64] = {};
}  // namespace

cudaError_t noalloc_scratch(float **ptr) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  const unsigned long long ctx = context_id();
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (g_noalloc_ptr[dev] == nullptr || ctx == 0 || g_noalloc_ctx[dev] != ctx) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_decode_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_noalloc_ptr[dev] = static_cast<float *>(p);
    g_noalloc_ctx[dev] = ctx;
  }
  *ptr = g_noalloc_ptr[dev];
  return cudaSuccess;
}

}  // namespace plx
