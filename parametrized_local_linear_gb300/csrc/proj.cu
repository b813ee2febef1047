// Fused input projection of a Parallax layer on the tcgen05 tensor cores:
//   [q | k | v | rho] = x [W_Q; W_K; W_V; W_R]^T
// with the probe rho_i = W_R x_i computed beside the usual projections
// ("Parallax: parametrized local linear attention for language modeling",
// section "Core mechanism"), bf16 operands, fp32 accumulation, and an
// epilogue that writes every output element straight into the per-head
// layouts the attention kernels read ([B, H, L, 128]).
//
// Persistent GEMM, one CTA per SM, in clusters of two that work as a CTA
// pair on the two-SM tensor-core form (tcgen05 .cta_group::2). A tile is 256
// token rows x 256 output features (two heads): each CTA of the pair loads
// its own 128 token rows of x and its half (128 rows) of the W tile, and the
// leader CTA issues 256 x 256 x 16 UMMAs that read A from both CTAs and B
// half from each, with the accumulator rows of each CTA in its own TMEM.
// Per SM a stage is then 32 KB of TMA writes and 32 KB of UMMA operand reads
// for 512 tensor cycles, 128 bytes per cycle: the single-SM form needed 192
// (a 48 KB stage written and read again) and ran the tensor pipe at most
// two-thirds busy, bound by shared-memory bandwidth. The K loop walks the
// model dimension in 64-element stages (one 128-byte swizzle atom) through a
// 6-stage TMA ring whose completion both CTAs count on the leader's
// barriers; the leader's UMMA commits release a stage in both CTAs. The two
// 256-column fp32 accumulators in TMEM alternate between tiles, so the
// epilogue of one tile overlaps the UMMAs of the next. 10 warps:
//   warp 0      TMA producer (x tile 128 x 64; this CTA's 128 W rows x 64)
//   warp 1      TMEM allocator (with the peer); in the leader one thread
//               issues the pair UMMAs
//   warps 2..9  epilogue, two warps per TMEM lane quarter, each with half
//               of the 256 columns: thread = token row = TMEM lane;
//               32-column chunks are converted to bf16 (round to nearest
//               even) and stored as 64 contiguous bytes of one head row.
//               With one warp per quarter the stores of a tile outlasted the
//               next tile's UMMAs at model dim 1024.
#include "plx_device.cuh"
#include "plx_internal.h"

namespace plx {
namespace {

constexpr int BM = 128, BN = 256, BK = 64, NST = 6, HD = 128;
constexpr int A_BYTES = BM * BK * 2;        // 16 KB: this CTA's 128 token rows
constexpr int B_BYTES = (BN / 2) * BK * 2;  // 16 KB: this CTA's half of the 256 W rows
constexpr int STAGE = A_BYTES + B_BYTES;    // 32 KB
constexpr int OFF_BAR = NST * STAGE;        // 196608
constexpr int NBAR = 2 * NST + 4 + 1;
constexpr int SMEM_BYTES = OFF_BAR + NBAR * 8 + 16 + 1024;
constexpr int EPI_WARPS = 8;
constexpr int THREADS = 32 * (2 + EPI_WARPS);

struct ProjArgs {
  __nv_bfloat16 *q, *k, *v, *r;
  int T, L, Hq, Hkv;     // tokens (B L), tokens per sequence, heads
  int mtp, npairs, kt;   // token-tile pairs, tile pairs (clusters' work units), K stages
  int D, F;              // model dim, stacked output features (2 Hq + 2 Hkv) d
  unsigned *err;
};

__global__ void __launch_bounds__(THREADS, 1)
    proj_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w,
                const ProjArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + OFF_BAR);
  uint64_t *full = bars;                // [NST] leader: both CTAs' parts of the stage loaded
  uint64_t *empty = full + NST;         // [NST] the pair UMMAs are done with the stage
  uint64_t *acc_full = empty + NST;     // [2] accumulator complete
  uint64_t *acc_empty = acc_full + 2;   // [2] leader: both CTAs' epilogue threads read it
  uint64_t *drain = acc_empty + 2;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + NBAR);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < NST; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), 1);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(smem_u32(&acc_full[x]), 1);
      mbar_init(smem_u32(&acc_empty[x]), 2 * 32 * EPI_WARPS);
    }
    mbar_init(smem_u32(drain), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tensormap(&tm_x);
    prefetch_tensormap(&tm_w);
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(tmem_slot), 512);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  // Both CTAs' barriers must be initialised before either signals the other.
  cluster_sync_all();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;
  const Abort ab{abort_flag, a.err};
  const int crank = static_cast<int>(cluster_ctarank());
  const bool leader = crank == 0;
  const int cid = blockIdx.x >> 1, ncl = gridDim.x >> 1;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ producer
      int g = 0, issued = 0;
      bool ok = true;
      for (int tp = cid; ok && tp < a.npairs; tp += ncl) {
        const int m0 = (2 * (tp % a.mtp) + crank) * BM, n0 = (tp / a.mtp) * BN;
        for (int kk = 0; kk < a.kt; ++kk, ++g) {
          const int st = g % NST;
          if (g >= NST && !mbar_wait(smem_u32(&empty[st]), ((g / NST) - 1) & 1, ab)) { ok = false; break; }
          // The W box lies inside W's rows and both boxes inside the model dim
          // (x rows past the tokens are zero-filled by TMA).
          if (!PLX_IN_BOUNDS(kk * BK < a.D && n0 + crank * (BN / 2) < a.F, ab)) { ok = false; break; }
          // The leader's barrier counts both CTAs' 32 KB.
          if (leader) mbar_arrive_expect_tx(smem_u32(&full[st]), 2 * STAGE);
          const uint32_t fb = mapa_shared(smem_u32(&full[st]), 0);
          const uint32_t base = smem_u32(smem + st * STAGE);
          tma_load_3d_pair(base, &tm_x, kk * BK, m0, 0, fb);
          tma_load_3d_pair(base + A_BYTES, &tm_w, kk * BK, n0 + crank * (BN / 2), 0, fb);
          issued = g + 1;
        }
      }
      // Only the leader can wait on the stage barriers; they count the
      // peer's copies too, and the peer waits for the leader at the end.
      if (ab.raised() && leader)
        for (int x = max(0, issued - NST); x < issued; ++x)
          mbar_wait_drain(smem_u32(&full[x % NST]), (x / NST) & 1);
    }
  } else if (warp == 1) {
    if (lane == 0 && leader) {
      // ------------------------------------------------------------ UMMA issuer
      constexpr uint32_t idesc = idesc_bf16_f32(2 * BM, BN, 0);
      const uint64_t adesc0 = smem_desc_sw128(smem_u32(smem), 16, 1024);
      const uint64_t bdesc0 = smem_desc_sw128(smem_u32(smem + A_BYTES), 16, 1024);
      int g = 0, it = 0;
      bool ok = true;
      for (int tp = cid; ok && tp < a.npairs; tp += ncl, ++it) {
        const int buf = it & 1;
        // The accumulator's previous tile must have been read out by both CTAs.
        if (it >= 2 && !mbar_wait(smem_u32(&acc_empty[buf]), ((it >> 1) - 1) & 1, ab)) break;
        tc_fence_after();
        const uint32_t d = tbase + buf * BN;
        for (int kk = 0; kk < a.kt; ++kk, ++g) {
          const int st = g % NST;
          if (!mbar_wait(smem_u32(&full[st]), (g / NST) & 1, ab)) { ok = false; break; }
          tc_fence_after();
          const uint64_t ad = adesc0 + st * (STAGE >> 4), bd = bdesc0 + st * (STAGE >> 4);
#pragma unroll
          for (int ks = 0; ks < BK / 16; ++ks)
            umma_ss_pair(d, ad + ks * 2, bd + ks * 2, idesc, (kk > 0 || ks > 0));
          umma_commit_pair_mc(smem_u32(&empty[st]), 0x3);  // release the stage in both CTAs
        }
        if (ok) umma_commit_pair_mc(smem_u32(&acc_full[buf]), 0x3);
      }
      umma_commit_pair_mc(smem_u32(drain), 0x1);
      mbar_wait_drain(smem_u32(drain), 0);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int qw = warp & 3, row = qw * 32 + lane;
    const int c0 = ((warp - 2) >> 2) * (BN / 64);  // first of this warp's 32-column chunks
    const uint32_t tl = tbase + (static_cast<uint32_t>(qw * 32) << 16);
    const int fq = a.Hq * HD, fk = fq + a.Hkv * HD, fv = fk + a.Hkv * HD;
    int it = 0;
    for (int tp = cid; tp < a.npairs; tp += ncl, ++it) {
      const int buf = it & 1;
      const bool ok = mbar_wait(smem_u32(&acc_full[buf]), (it >> 1) & 1, ab);
      if (!__all_sync(0xffffffffu, ok)) break;
      tc_fence_after();
      const int m0 = (2 * (tp % a.mtp) + crank) * BM, n0 = (tp / a.mtp) * BN;
      const int t = m0 + row;
      const bool valid = t < a.T;
      const int b = valid ? t / a.L : 0, l = valid ? t - b * a.L : 0;
#pragma unroll 1
      for (int c = c0; c < c0 + BN / 64; ++c) {
        float vals[32];
        tmem_ld32(tl + buf * BN + c * 32, vals);
        tmem_wait_ld();
        // Feature f of the stacked output: which projection, head, column.
        const int f = n0 + c * 32;
        __nv_bfloat16 *dst;
        int H, fo;
        if (f < fq) { dst = a.q; H = a.Hq; fo = f; }
        else if (f < fk) { dst = a.k; H = a.Hkv; fo = f - fq; }
        else if (f < fv) { dst = a.v; H = a.Hkv; fo = f - fk; }
        else { dst = a.r; H = a.Hq; fo = f - fv; }
        if (valid && PLX_IN_BOUNDS(fo / HD < H && fo % HD + 32 <= HD && f < a.F, ab)) {
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 32; e += 2) pk[e >> 1] = pack_bf16x2(vals[e], vals[e + 1]);
          const int h = fo / HD, col = fo % HD;
          uint4 *d4 = reinterpret_cast<uint4 *>(
              dst + ((static_cast<size_t>(b) * H + h) * a.L + l) * HD + col);
#pragma unroll
          for (int u = 0; u < 4; ++u) d4[u] = make_uint4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
        }
      }
      tc_fence_before();
      mbar_arrive_cluster(mapa_shared(smem_u32(&acc_empty[buf]), 0));
    }
  }

  tc_fence_before();
  __syncthreads();
  // Every pair UMMA has completed (the leader drained them; the peer's
  // epilogue saw the last accumulator) once both CTAs are here.
  cluster_sync_all();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tbase, 512);
  }
  // Neither CTA leaves while the other may still signal its barriers.
  cluster_sync_all();
}

// 2-D bf16 map over [rows][cols] (cols contiguous) as a 3-D map with one
// plane; boxes of box_rows x 64, 128-byte swizzle, zero fill outside.
bool make_rows_map(EncodeTiledFn enc, CUtensorMap *map, const void *ptr, long long rows, int cols,
                   int box_rows) {
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows), 1};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(cols) * 2,
                                 static_cast<cuuint64_t>(rows) * cols * 2};
  const cuuint32_t box[3] = {BK, static_cast<cuuint32_t>(box_rows), 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(ptr), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_qkvr_proj(const void *x, const void *w, void *q, void *k, void *v, void *r,
                             int B, int L, int D, int Hq, int Hkv, unsigned *err,
                             cudaStream_t stream) {
  static thread_local unsigned long long configured_ctx = 0;
  const unsigned long long ctx = context_id();
  if (ctx == 0 || configured_ctx != ctx) {
    cudaError_t e = cudaFuncSetAttribute(proj_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         SMEM_BYTES);
    if (e != cudaSuccess) return e;
    configured_ctx = ctx;
  }
  EncodeTiledFn enc = encode_tiled_fn();
  if (enc == nullptr) return cudaErrorInvalidValue;
  const long long T = static_cast<long long>(B) * L;
  const int F = (2 * Hq + 2 * Hkv) * HD;
  CUtensorMap mx, mw;
  if (!make_rows_map(enc, &mx, x, T, D, BM) || !make_rows_map(enc, &mw, w, F, D, BN / 2))
    return cudaErrorInvalidValue;
  ProjArgs a;
  a.q = static_cast<__nv_bfloat16 *>(q);
  a.k = static_cast<__nv_bfloat16 *>(k);
  a.v = static_cast<__nv_bfloat16 *>(v);
  a.r = static_cast<__nv_bfloat16 *>(r);
  a.T = static_cast<int>(T);
  a.L = L;
  a.Hq = Hq;
  a.Hkv = Hkv;
  const int mt = static_cast<int>((T + BM - 1) / BM);
  a.mtp = (mt + 1) / 2;  // an odd last tile's partner reads zero rows and stores nothing
  a.npairs = a.mtp * (F / BN);  // F = 256 (Hq + Hkv): whole feature tiles
  a.kt = (D + BK - 1) / BK;
  a.D = D;
  a.F = F;
  a.err = err;
  const int clusters = min(a.npairs, sm_count() / 2);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * clusters);
  cfg.blockDim = dim3(THREADS);
  cfg.dynamicSmemBytes = SMEM_BYTES;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, proj_kernel, mx, mw, a);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace plx
