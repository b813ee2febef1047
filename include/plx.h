/*
 * plx.h -- C ABI of libplx.so, the GB300 (sm_103a) Parallax attention forward.
 *
 * Parallax ("Parallax: parametrized local linear attention for language
 * modeling", section "Core mechanism", output equation) corrects causal
 * softmax attention by the softmax-weighted KV cross-covariance seen by each
 * query, probed by a learned per-query vector rho_i = W_R x_i:
 *
 *     o_i = o^SA_i - Sigma_KV^(i) rho_i
 *     w_ij = softmax_j(q_i . k_j / sqrt(d)),   o^SA_i = sum_j w_ij v_j
 *     Sigma_KV^(i) = sum_j w_ij (v_j - o^SA_i)(k_j - mu_i)^T,  mu_i = sum_j w_ij k_j
 *
 * The kernels never form Sigma. They stream the keys once, as the pages'
 * FlashAttention-compatible streaming algorithm (section "Hardware-aware
 * algorithm") does, using the exact identity
 *
 *     o = O1 - O2 + O1 * s,  T_ij = rho_i . k_j,  O1 = P V,  O2 = (P o T) V,
 *     s = rowsum(P o T)      (P the softmax weights)
 *
 * which follows because sum_j w_ij (v_j - o^SA_i) = 0 removes the mu term.
 *
 * Conventions shared by every entry point
 *   - All tensor pointers are DEVICE pointers owned by the caller; the library
 *     keeps no reference after the call returns. Every call is asynchronous
 *     and ordered on `stream` (a cudaStream_t; NULL = legacy default stream).
 *   - Tensors are dense and contiguous, head dimension d innermost.
 *   - Query head h reads KV head h / (Hq / Hkv) (consecutive grouping, GQA).
 *   - Softmax scale is 1/sqrt(d); causal masking keeps keys j <= i; T uses
 *     the raw keys (any scale of the probe lives in W_R).
 *   - Inputs must be finite. A gate on the correction branch is applied by
 *     the caller by scaling r (the correction is linear in rho).
 *   - Arguments are validated on the host before any launch; a rejected call
 *     launches nothing and returns PLX_ERR_INVALID_ARG or PLX_ERR_UNSUPPORTED.
 *     plx_last_error_message() then says which argument was wrong.
 *   - Every wait inside a kernel is bounded. A wait that runs out sets a
 *     device error word instead of hanging; plx_check_device_error() reads
 *     (and clears) it and returns PLX_ERR_DEVICE_TIMEOUT.
 */
#ifndef PLX_H
#define PLX_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int plx_status;

#define PLX_OK 0
#define PLX_ERR_INVALID_ARG 1    /* null / misaligned pointer, bad size or ratio */
#define PLX_ERR_UNSUPPORTED 2    /* valid but not implemented (e.g. head dim) */
#define PLX_ERR_CUDA 3           /* a CUDA runtime or driver call failed */
#define PLX_ERR_DEVICE_TIMEOUT 4 /* a bounded in-kernel wait ran out */
#define PLX_ERR_BOUNDS 5         /* a device-side index check failed (debug build only) */

/*
 * Causal prefill, bf16 in / bf16 out, fp32 accumulation (tcgen05 tensor cores).
 *   q, r  : bf16 [B, Hq, L, d]   queries and probes rho (one probe per query head)
 *   k, v  : bf16 [B, Hkv, L, d]
 *   out   : bf16 [B, Hq, L, d]   o = o^SA - Sigma_KV rho, rounded to nearest even
 *   lse   : fp32 [B, Hq, L]      natural-log log-sum-exp of the scaled scores;
 *                                may be NULL
 *   d must be 128; Hq % Hkv == 0; B, Hq, Hkv, L >= 1; every pointer 16-byte
 *   aligned (TMA). Requires an sm_100-family GPU with tcgen05 (sm_103a build).
 */
plx_status plx_prefill_fwd(const void *q, const void *k, const void *v, const void *r,
                           void *out, float *lse, int B, int Hq, int Hkv, int L, int d,
                           void *stream);

/*
 * Chunked causal prefill: Lq new queries against Lk >= Lq keys of which they
 * are the last Lq positions (a chunk appended to an existing cache, the
 * cache already holding the chunk's own keys). Query row i sees keys
 * 0 .. Lk - Lq + i. Same dtypes and rules as plx_prefill_fwd; layouts:
 *   q, r, out : bf16 [B, Hq, Lq, d];   k, v : bf16 [B, Hkv, Lk, d];
 *   lse       : fp32 [B, Hq, Lq] or NULL.
 * plx_prefill_fwd is this call with Lq = Lk = L. The pages do not describe
 * chunked prefill; it is the serving form of the same causal forward.
 */
plx_status plx_prefill_fwd_chunk(const void *q, const void *k, const void *v, const void *r,
                                 void *out, float *lse, int B, int Hq, int Hkv, int Lq, int Lk,
                                 int d, void *stream);

/*
 * Chunked prefill with a per-row side output: the correction-to-output ratio
 * COR, which the page "Parallax: parametrized local linear attention for
 * language modeling" reports per layer in its experimental results (optimizer
 * dependence) without giving a formula. Reading used here, per query row:
 *   cor = |Sigma_KV rho| / |o|   (Euclidean norms over the d values of the
 *                                 fp32 correction and output before the bf16
 *                                 rounding of o; 0 when |o| = 0)
 * Arguments, layouts and results as plx_prefill_fwd_chunk, plus
 *   cor : fp32 [B, Hq, Lq], must not be NULL.
 * A per-layer COR is the mean (or any other statistic) of cor over rows,
 * taken by the caller.
 */
plx_status plx_prefill_fwd_cor(const void *q, const void *k, const void *v, const void *r,
                               void *out, float *lse, float *cor, int B, int Hq, int Hkv, int Lq,
                               int Lk, int d, void *stream);

/*
 * Training forward: plx_prefill_fwd (Lq = Lk = L) that also saves what the
 * backward pass needs. Extra outputs, none of which may be NULL:
 *   lse  : fp32 [B, Hq, L]     as plx_prefill_fwd
 *   o1   : bf16 [B, Hq, L, d]  o^SA, the softmax attention output per row
 *   sbar : fp32 [B, Hq, L]     sum_j w_j (rho . k_j), the softmax-weighted
 *                              mean of the probe-key products per row
 * o is identical bit for bit to plx_prefill_fwd's.
 */
plx_status plx_prefill_fwd_train(const void *q, const void *k, const void *v, const void *r,
                                 void *out, float *lse, void *o1, float *sbar, int B, int Hq,
                                 int Hkv, int L, int d, void *stream);

/*
 * Backward pass of the causal prefill: the gradients of sum(dout * o) with
 * respect to q, k, v and rho. The pages ("Parallax: parametrized local linear
 * attention for language modeling") train with this layer but print no
 * backward pass; the gradient is that of the forward definition (section
 * "Core mechanism", output equation), streamed over the causal pairs with
 * the forward's saved lse, o^SA and sbar.
 *   q, r, out, o1, dout : bf16 [B, Hq, L, d]   (out, o1 from plx_prefill_fwd_train)
 *   k, v                : bf16 [B, Hkv, L, d]
 *   lse, sbar           : fp32 [B, Hq, L]      (from plx_prefill_fwd_train)
 *   dq, dr              : bf16 [B, Hq, L, d]   written
 *   dk, dv              : bf16 [B, Hkv, L, d]  written (summed over each
 *                                              kv head's query heads)
 * d must be 128; every pointer non-NULL and 16-byte aligned. Allocates a
 * stream-ordered workspace of B * Hq * round_up(L, 64) * 16 bytes
 * (cudaMallocAsync / cudaFreeAsync on `stream`). Deterministic: no atomics,
 * every output row is written by one thread block.
 */
plx_status plx_prefill_bwd(const void *q, const void *k, const void *v, const void *r,
                           const void *out, const void *o1, const float *lse, const float *sbar,
                           const void *dout, void *dq, void *dk, void *dv, void *dr, int B, int Hq,
                           int Hkv, int L, int d, void *stream);

/*
 * Fused input projection of a Parallax layer: q, k, v and the probe
 * rho = W_R x (page "Parallax: parametrized local linear attention for
 * language modeling", section "Core mechanism") from one product
 *   y = x [W_Q; W_K; W_V; W_R]^T,
 * written straight into the per-head layouts the attention calls take.
 *   x : bf16 [B * L, D]                 token rows; sequence b at rows b L ..
 *   w : bf16 [(2 Hq + 2 Hkv) d, D]      rows W_Q (Hq d), W_K (Hkv d),
 *                                       W_V (Hkv d), W_R (Hq d); each
 *                                       part's rows grouped by head
 *   q, r : bf16 [B, Hq, L, d];   k, v : bf16 [B, Hkv, L, d]   written
 * fp32 accumulation, outputs rounded to nearest even. d must be 128, D a
 * positive multiple of 8; every pointer 16-byte aligned. W_R = 0 (the pages'
 * start for adapting a pretrained model) gives rho = 0 exactly, and the
 * layer is then softmax attention.
 */
plx_status plx_qkvr_proj(const void *x, const void *w, void *q, void *k, void *v, void *r, int B,
                         int L, int D, int Hq, int Hkv, int d, void *stream);

/*
 * Causal prefill in fp32 (CUDA cores, fp32 arithmetic throughout). Same
 * arguments and layouts as plx_prefill_fwd with float tensors; d in {64, 128}.
 * This is the exact-arithmetic path used to check parity at 1e-5 relative error.
 */
plx_status plx_prefill_fwd_f32(const float *q, const float *k, const float *v, const float *r,
                               float *out, float *lse, int B, int Hq, int Hkv, int L, int d,
                               void *stream);

/*
 * Decode: one new query per sequence against its KV cache, bf16 in / out,
 * fp32 accumulation ("Parallax: parametrized local linear attention for
 * language modeling", sections "Core mechanism" and "Hardware-aware
 * algorithm": the covariance branch reads the same key and value stream as
 * the softmax branch).
 *   q, r           : bf16 [B, Hq, d]
 *   kcache, vcache : bf16 packed [sum_b seqlens[b], Hkv, d]; sequence b starts
 *                    at token sum_{b' < b} seqlens[b'], fewer than 2^30 tokens
 *                    in all. The cache already holds the current token: the
 *                    query sees all seqlens[b] keys.
 *   seqlens        : int32 [B] on the device, each >= 0. A sequence of length
 *                    0 gets an all-zero output row.
 *   out            : bf16 [B, Hq, d]
 *   d must be 128; Hq % Hkv == 0, Hq / Hkv <= 8 and B * Hq <= 2^24.
 * The keys of all sequences and kv heads form one stream that is cut into
 * equal shares, one CTA each, so a ragged batch keeps every CTA equally busy;
 * each CTA writes a partial record (log-sum-exp, normalised O1, O2, sigma)
 * per (sequence, query head) it meets, and a second kernel combines them.
 * The records go to a stream-ordered scratch buffer (cudaMallocAsync /
 * cudaFreeAsync on `stream`) of plx_decode_workspace_bytes(B, Hq, Hkv, d,
 * plx_decode_default_nsplit(B, Hkv)) bytes.
 */
plx_status plx_decode_fwd(const void *q, const void *r, const void *kcache, const void *vcache,
                          const int *seqlens, void *out, int B, int Hq, int Hkv, int d,
                          void *stream);

/*
 * plx_decode_fwd with an explicit number of shares, nsplit >= 1 (one CTA
 * each; share c of n holds the keys [floor(c W / n), floor((c + 1) W / n)) of
 * the W keys of the batch, sequence-major, then kv head, then token; at most
 * W shares take part), and a caller-provided device workspace of at least
 * plx_decode_workspace_bytes(B, Hq, Hkv, d, nsplit) bytes, 16-byte aligned.
 * nsplit <= 0 picks the default schedule: floor(sqrt(W)) shares, at most
 * plx_decode_default_nsplit (small batches get fewer, shorter shares); when
 * all sequences of nonzero length have one length, at most 256, lowered to a
 * count that cuts every (sequence, kv head) row at the same keys or gives
 * every share whole rows, if that keeps at least 80% of the shares.
 * workspace == NULL allocates as plx_decode_fwd does. The result does not
 * depend on nsplit beyond fp32 rounding.
 */
plx_status plx_decode_fwd_ex(const void *q, const void *r, const void *kcache, const void *vcache,
                             const int *seqlens, void *out, int B, int Hq, int Hkv, int d,
                             int nsplit, void *workspace, size_t workspace_bytes, void *stream);

/*
 * Decode with the per-(sequence, head) correction-to-output ratio (see
 * plx_prefill_fwd_cor for the reading): arguments, layouts, allocation and
 * results as plx_decode_fwd, plus
 *   cor : fp32 [B, Hq], must not be NULL; 0 for sequences of length 0.
 * The ratio is formed after the partial records are combined, from the
 * combined fp32 correction and output.
 */
plx_status plx_decode_fwd_cor(const void *q, const void *r, const void *kcache, const void *vcache,
                              const int *seqlens, void *out, float *cor, int B, int Hq, int Hkv,
                              int d, void *stream);

/*
 * plx_decode_fwd for callers that cannot allocate device memory during the
 * call: for example code whose device memory belongs to an allocator that
 * must not be bypassed, a host thread that must not take the driver's
 * allocation locks, or an embedding that gives this library only its own
 * input and output buffers. There is no counterpart in the
 * paper; it exists for such callers only. Same arguments, layouts and results
 * as plx_decode_fwd; the partial records go to one fixed device array of
 * 16 MiB that the library reserves on every device that loads it, held until
 * the process exits. Nothing is allocated or freed by this call.
 *   - The schedule is the default one, with fewer shares if needed so the
 *     records fit; plx_decode_workspace_bytes(B, Hq, Hkv, d, 1) must fit in
 *     16 MiB, else PLX_ERR_UNSUPPORTED and nothing runs.
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress); make that first call before any stream capture.
 *     The address is kept per device together with the id of the CUDA
 *     context it belongs to; after a cudaDeviceReset the next call runs in a
 *     new context and looks the address up again (outside a capture too).
 *   - Every call shares the array: calls that overlap on the GPU race and must
 *     be serialised by the caller. The array needs no clearing between calls
 *     (each call writes every record it reads).
 */
plx_status plx_decode_fwd_noalloc(const void *q, const void *r, const void *kcache,
                                  const void *vcache, const int *seqlens, void *out, int B, int Hq,
                                  int Hkv, int d, void *stream);

/* Bytes of decode workspace for nsplit shares: a table of 8 bytes per
 * (sequence, kv head) rounded up to 256 bytes, then
 * (nsplit * Hq / Hkv + B * Hq) fp32 records of 2 d + 2 floats. 0 for
 * arguments out of range. */
size_t plx_decode_workspace_bytes(int B, int Hq, int Hkv, int d, int nsplit);

/* The number of shares plx_decode_fwd starts from on the current device: two
 * CTAs per SM, one wave of the split kernel (B and Hkv do not change it; the
 * kernel itself uses fewer for small batches, since lengths are on the device). */
int plx_decode_default_nsplit(int B, int Hkv);

/* Synchronises `stream`, then reads and clears the device error word.
 * PLX_ERR_DEVICE_TIMEOUT if a bounded wait ran out since the last check,
 * PLX_ERR_INVALID_ARG if a kernel found its device-side inputs out of range
 * (decode lengths summing to 2^30 tokens or more; that call did no work and
 * its outputs are undefined), PLX_ERR_BOUNDS if a device-side index check of
 * a debug build failed (below), PLX_ERR_CUDA if the stream reports an error,
 * else PLX_OK.
 *
 * Debug build: the same sources compiled with PLX_DEBUG_BOUNDS
 * (python -m parametrized_local_linear_gb300.build --debug-bounds, giving
 * libplx_debug.so with this same interface) check, before each TMA copy and
 * each indexed global store, that the coordinates or index lie inside the
 * buffer: the tensor-map coordinates of every prefill, backward and
 * projection box, every decode box against its sequence's tokens, and the
 * decode's query rows and record slots. A failed check skips the access,
 * stops the CTA as a timed-out wait does and sets the bit that this call
 * reports as PLX_ERR_BOUNDS; nothing traps. Outputs of a call that passed
 * every check equal the release library's bit for bit. */
plx_status plx_check_device_error(void *stream);

/* Launches one block whose wait on an mbarrier that nothing ever arrives on
 * runs out after about `limit_cycles` SM clock cycles; the kernel then sets
 * the device error word and returns. Exercises the failure path of the
 * bounded waits without faulting or hanging the GPU. */
plx_status plx_debug_timeout_probe(long long limit_cycles, void *stream);

/* Static description of a status code. */
const char *plx_status_string(plx_status s);

/* Detail of the last non-OK status returned on the calling host thread. */
const char *plx_last_error_message(void);

#ifdef __cplusplus
}
#endif

#endif /* PLX_H */
