/*
 * attn.h -- C interface of libattn.so: exact fused attention forward with
 * online softmax, and split-KV decode, on NVIDIA GB300 (sm_103a).
 *
 * The operation (all entry points):
 *   For every batch b, head h and query row i, over the keys j visible
 *   from i (mask below):
 *     s_j   = scale * <q_i, k_j>
 *     o_i   = sum_j softmax(s)_j v_j
 *     lse_i = m + log(l), m = max_j s_j, l = sum_j exp(s_j - m)
 *   Source pages:
 *     P1 "Derive online softmax, prove it is exact, and explain why it makes
 *        FlashAttention fast without reducing FLOPs"
 *        (inferenceinterviews.com/q/online-softmax-derive-and-prove-flashattention):
 *        "A strong answer" -- softmax attention for one query, the block
 *        recurrence for (m, l, a), o = a / l exact; "What interviewers probe
 *        next" -- the per-row log-sum-exp m + log l kept for the backward
 *        pass, and split-KV (Flash-Decoding) for batch-1 long-context decode.
 *     P2 "Implement online softmax for a whole tile of queries, not one
 *        query, and write the rescaling step in matrix form"
 *        (inferenceinterviews.com/q/online-softmax-query-tile-matrix-form):
 *        "A strong answer" -- the query-tile equations S_j, m', P_j, l', A',
 *        alpha and the single diag(l)^-1 at the end; the m_ref guard for rows
 *        that see no key; causal masking by absolute position.
 *     P3 "Online softmax" (interview.clozo.ai/blog/online-softmax.html):
 *        "Step 4" -- the associative merge of partial results; "Trade-offs
 *        and edge cases" -- Flash-Decoding's per-chunk log-sum-exp and final
 *        rescaling reduction.
 *
 * Conventions shared by every entry point:
 *   - All tensor pointers are DEVICE pointers, contiguous, row-major:
 *     q [B,H,Nq,d], k and v [B,H,Nk,d], o [B,H,Nq,d], lse [B,H,Nq] (FP32,
 *     natural log). Every tensor pointer must be 16-byte aligned.
 *   - Masks (mask_kind, bit flags, combined by AND):
 *       ATTN_MASK_CAUSAL  key j visible from query i iff j <= i (query i and
 *                         key j at their own indices: top-left alignment).
 *       ATTN_MASK_WINDOW  sliding window of `window` keys ending at the
 *                         query: visible iff i - window < j <= i (implies the
 *                         causal bound); window >= 1.
 *       ATTN_MASK_PADDING keys j >= seqlens_k[b] invisible; seqlens_k is a
 *                         device int32 [B] array, values clamped to [0, Nk].
 *   - A row with no visible key gets o = 0 and lse = -inf (never NaN).
 *   - Ownership: the caller allocates every buffer (including the decode
 *     workspace); the library allocates no device memory on these paths and
 *     keeps no state between calls except a per-device error word.
 *   - The library looks up the device addresses of its own device variables
 *     (the error word, and the fixed array of attn_decode_splitkv_noalloc)
 *     once per device and keeps them for the life of the process. Resetting
 *     a device (cudaDeviceReset) or destroying its primary context while the
 *     library is loaded makes those addresses stale; that is not supported.
 *   - Calls are asynchronous and stream-ordered on `stream` (0 = legacy
 *     default stream). Argument errors are reported synchronously by the
 *     return value, with a message in attn_last_error(); the outputs are then
 *     untouched. A kernel whose bounded wait expired reports it through
 *     attn_check_device_error().
 *   - Supported head dims: d in {64, 128}; anything else is
 *     ATTN_ERR_UNSUPPORTED.
 */
#ifndef ATTN_H_
#define ATTN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    ATTN_OK = 0,
    ATTN_ERR_INVALID_ARG = 1,   /* null/misaligned pointer, bad size or flag */
    ATTN_ERR_UNSUPPORTED = 2,   /* valid but not implemented (e.g. d = 96)   */
    ATTN_ERR_CUDA = 3,          /* a CUDA runtime/driver call failed         */
    ATTN_ERR_TIMEOUT = 4        /* a device-side bounded wait expired        */
} attn_status_t;

enum {
    ATTN_MASK_NONE = 0,
    ATTN_MASK_CAUSAL = 1,
    ATTN_MASK_WINDOW = 2,
    ATTN_MASK_PADDING = 4
};

/* Element types of attn_softmax_rows. */
enum {
    ATTN_DTYPE_F32 = 0,
    ATTN_DTYPE_BF16 = 1
};

/* Opaque CUDA stream handle (cudaStream_t / CUstream). */
typedef void* attn_stream_t;

/*
 * attn_fwd -- fused attention forward, BF16 inputs and output.
 *
 * Computes o and lse as defined above for q, k, v in BF16 (o in BF16, lse in
 * FP32). Query tiles of 128 rows stream 128-key blocks of K and V through
 * shared memory; the running row max m, normalizer l and unnormalised
 * accumulator A stay on chip (A in tensor memory), updated per block as
 * A <- diag(alpha) A + P V with alpha = exp(m_old - m_new) (P2 "A strong
 * answer"), with one diag(l)^-1 at the end; the score matrix never reaches
 * device memory. P is rounded to BF16 for the P V product; m, l and A are
 * FP32. Blocks that the mask hides entirely are skipped before they are
 * loaded (P1 "Common mistakes", on causal masking).
 *
 *   q, k, v      device BF16 pointers, layout above.
 *   o            device BF16 [B,H,Nq,d] (written).
 *   lse          device FP32 [B,H,Nq] (written); may be NULL to skip it.
 *   B, H         batch and heads, >= 0.
 *   Nq, Nk       query and key lengths, >= 0 (Nk = 0: every row is empty).
 *   d            head dimension, 64 or 128.
 *   scale        score scale (usually 1/sqrt(d)); finite and > 0.
 *   mask_kind    OR of ATTN_MASK_* flags.
 *   window       window length (>= 1) when ATTN_MASK_WINDOW is set.
 *   seqlens_k    device int32 [B], required iff ATTN_MASK_PADDING is set.
 *   stream       CUDA stream.
 */
attn_status_t attn_fwd(const void* q, const void* k, const void* v,
                       void* o, float* lse,
                       int B, int H, int Nq, int Nk, int d, float scale,
                       int mask_kind, int window, const int* seqlens_k,
                       attn_stream_t stream);

/*
 * attn_fwd_host_workspace_bytes -- size in bytes of the device workspace that
 * attn_fwd_host needs: min(slots, number of groups) buffer sets, each
 * holding q, k, v, o (BF16) and lse (FP32) for ceil(B*H / groups) heads,
 * plus the per-head key lengths, at 256-byte-aligned offsets. Returns 0 for
 * invalid arguments (negative sizes, d not in {64, 128}, groups < 1, slots
 * outside [1, 8]).
 */
size_t attn_fwd_host_workspace_bytes(int B, int H, int Nq, int Nk, int d, int groups,
                                     int slots);

/*
 * attn_fwd_host_groups -- the number of head groups (one forward kernel
 * launch each) attn_fwd_host uses for B*H heads and `groups`: the group
 * sizes are described there. Returns -1 for negative sizes or groups < 1,
 * 0 when B*H is 0. Host-only; never touches the device.
 */
int attn_fwd_host_groups(int B, int H, int groups);

/*
 * attn_fwd_host -- attn_fwd for inputs and outputs in HOST memory.
 *
 * Only Q, K, V and O cross device memory in the fused method (P1 "Derive
 * online softmax, ...", "A strong answer", the cost paragraph); this call
 * moves exactly those across the host link, overlapped with the kernel. The
 * B*H heads are cut into contiguous groups of at most P = ceil(B*H / groups)
 * heads: groups of P heads, except that when B*H >= 4 P (and P >= 4) the
 * first two groups have ceil(P/4) and ceil(P/2) heads and the last two
 * ceil(P/2) and ceil(P/4), so that the first kernel starts after a short
 * copy and the last copy-back follows a short kernel
 * (attn_fwd_host_groups gives the count). Group g is copied into buffer
 * set g % slots of the workspace (one
 * cudaMemcpyAsync per tensor), computed by the attn_fwd kernel on that
 * slot's stream, and its o and lse copied back, so that the copy-in of one
 * group, the kernel of the next and the copy-out of the previous run at the
 * same time. A slot is refilled once its previous group has been copied
 * out. The result is bit for bit that of attn_fwd on the same values.
 *
 *   q, k, v      HOST BF16 pointers, [B,H,Nq,d] and [B,H,Nk,d], 2-byte
 *                aligned. Page-locked memory (cudaHostAlloc /
 *                cudaHostRegister) is needed for the copies to overlap the
 *                kernels; pageable memory works but serialises them.
 *   o            HOST BF16 [B,H,Nq,d] (written).
 *   lse          HOST FP32 [B,H,Nq] (written), or NULL.
 *   B..window    as attn_fwd.
 *   seqlens_k    HOST int32 [B], required iff ATTN_MASK_PADDING is set.
 *   groups       number of head groups, >= 1 (more than B*H acts as B*H).
 *   slots        device buffer sets in flight, 1..8 (3 keeps the copy-in
 *                stream busy on a ~200 GB/s host link).
 *   workspace    caller-owned DEVICE buffer of at least
 *                attn_fwd_host_workspace_bytes(B, H, Nq, Nk, d, groups,
 *                slots) bytes, 256-byte aligned; overwritten. Two calls that
 *                share a workspace must be ordered on one stream.
 *   stream       the caller's stream: the copies and kernels start after the
 *                work already queued on it, and work queued on it after this
 *                call starts once o and lse are in host memory. The call
 *                returns once everything is queued; synchronise `stream`
 *                before reading o or lse, and keep every host buffer,
 *                seqlens_k included, alive and unmodified until then.
 * The library creates, on the first call on a device, two copy streams,
 * eight compute streams and their events, and keeps them for the life of
 * the process; calls on one device are queued one at a time. No device
 * memory is allocated. Errors: as attn_fwd, plus ATTN_ERR_INVALID_ARG for a
 * missing or short workspace or bad groups/slots; a CUDA error while
 * queueing returns ATTN_ERR_CUDA with part of the work queued.
 */
attn_status_t attn_fwd_host(const void* q, const void* k, const void* v,
                            void* o, float* lse,
                            int B, int H, int Nq, int Nk, int d, float scale,
                            int mask_kind, int window, const int* seqlens_k,
                            int groups, int slots, void* workspace, size_t workspace_bytes,
                            attn_stream_t stream);

/*
 * attn_fwd_fp8 -- attn_fwd with 8-bit floating-point inputs, the FP8 mode P1
 * ("What did FlashAttention-2 and -3 change?") and P3 ("Where the merge is
 * used today") credit to FlashAttention-3. q, k and v hold E4M3 values
 * (1 sign, 4 exponent, 3 mantissa bits, bias 7, no infinities; one byte
 * each, layout as attn_fwd); the real inputs are q*descale_q, k*descale_k
 * and v*descale_v, per-tensor factors chosen by the caller when quantising.
 * Computed: O = softmax(scale * Q K^T + mask) V and lse on those real
 * values, with both products on the 8-bit tensor-core path (FP32
 * accumulation) and the attention weights rounded to E4M3 for the P V
 * product; the row sums l, the running maxima and the accumulator are FP32.
 *
 *   q, k, v      device E4M3 pointers, [B,H,N,128], 16-byte aligned.
 *   o            device BF16 [B,H,Nq,128] (written).
 *   lse          device FP32 [B,H,Nq] (written), natural log of the real
 *                scores' sum of exponentials; may be NULL.
 *   d            must be 128 (ATTN_ERR_UNSUPPORTED otherwise).
 *   descale_*    finite and > 0; scale * descale_q * descale_k * log2(e)
 *                must be finite in FP32.
 *   others       as attn_fwd (masks, empty rows, errors, stream).
 */
attn_status_t attn_fwd_fp8(const void* q, const void* k, const void* v,
                           void* o, float* lse,
                           int B, int H, int Nq, int Nk, int d, float scale,
                           float descale_q, float descale_k, float descale_v,
                           int mask_kind, int window, const int* seqlens_k,
                           attn_stream_t stream);

/*
 * attn_fwd_f32 -- the same operation with FP32 q, k, v and o (lse FP32).
 * All arithmetic is FP32 on the CUDA cores; intended for accuracy checks of
 * small problems such as P2's 1,000-key tile test. Arguments as attn_fwd.
 */
attn_status_t attn_fwd_f32(const float* q, const float* k, const float* v,
                           float* o, float* lse,
                           int B, int H, int Nq, int Nk, int d, float scale,
                           int mask_kind, int window, const int* seqlens_k,
                           attn_stream_t stream);

/*
 * attn_bwd_workspace_bytes -- bytes of scratch attn_bwd needs: two FP32
 * values (the row's log-sum-exp in log2 units and D = <dO, O>) per query
 * row, rows rounded up to a multiple of 128 per (b, h), in two 256-byte
 * aligned regions; at d = 128 also an FP32 dQ accumulator of d values per
 * such row (for B=1, H=64, Nq=8192: 256 MiB). Returns 0 for invalid
 * arguments.
 */
size_t attn_bwd_workspace_bytes(int B, int H, int Nq, int d);

/*
 * attn_bwd -- backward pass of attn_fwd, from the saved per-row log-sum-exp.
 *
 * The forward keeps only O and lse; the backward rebuilds the normalised
 * probabilities P = exp(S - lse) block by block with no running max (P1
 * "What interviewers probe next", on what the backward pass stores; P2
 * "A strong answer", closing paragraph). With D_i = <dO_i, O_i>:
 *   dV = P^T dO,  dS = P * (dO V^T - D),  dQ = scale dS K,  dK = scale dS^T Q.
 * Three launches on `stream`. d = 128: D and lse into the workspace (and
 * the dQ accumulator zeroed); a keys-outer kernel accumulating dK and dV in
 * tensor memory and adding each key block's dQ contribution into the FP32
 * accumulator in the workspace; dQ = scale * accumulator to BF16. The order
 * of those additions is not fixed, so dQ may differ in its last bit between
 * runs (dK, dV are reproducible). d = 64: D and lse; the keys-outer kernel
 * for dK, dV; a queries-outer kernel for dQ (S and dP recomputed there).
 *
 *   q, k, v      device BF16, as for attn_fwd.
 *   o            device BF16 [B,H,Nq,d]: the forward output.
 *   dout         device BF16 [B,H,Nq,d]: gradient of the loss w.r.t. o.
 *   lse          device FP32 [B,H,Nq]: the forward log-sum-exp (natural
 *                log; -inf for rows with no visible key).
 *   dq           device BF16 [B,H,Nq,d] (written).
 *   dk, dv       device BF16 [B,H,Nk,d] (written; keys no query sees get 0).
 *   B..window, seqlens_k, stream: exactly the values the forward used.
 *   workspace    caller-owned device scratch of at least
 *                attn_bwd_workspace_bytes(B, H, Nq, d) bytes, 256-byte
 *                aligned; overwritten.
 * P and dS are rounded to BF16 for the tensor-core products; accumulation
 * is FP32. Errors: as attn_fwd; ATTN_ERR_INVALID_ARG for a missing or short
 * workspace.
 */
attn_status_t attn_bwd(const void* q, const void* k, const void* v, const void* o,
                       const void* dout, const float* lse, void* dq, void* dk, void* dv,
                       int B, int H, int Nq, int Nk, int d, float scale,
                       int mask_kind, int window, const int* seqlens_k,
                       void* workspace, size_t workspace_bytes, attn_stream_t stream);

/*
 * attn_decode_workspace_bytes -- size in bytes of the scratch buffer that
 * attn_decode_splitkv needs for (B, H, d, num_splits): per (b, h, split) one
 * FP32 partial output of d values and one FP32 partial log-sum-exp, at
 * 256-byte-aligned offsets. Returns 0 for invalid arguments.
 */
size_t attn_decode_workspace_bytes(int B, int H, int d, int num_splits);

/*
 * attn_decode_splitkv -- split-KV decode (Flash-Decoding): one query row per
 * (b, h), keys split into `num_splits` contiguous chunks of
 * ceil(Nk / num_splits) keys.
 *
 * Launch 1 runs the online recurrence of P1 "A strong answer" over each
 * chunk and writes the chunk's normalised output o_s and log-sum-exp lse_s
 * to the workspace (an empty chunk writes o_s = 0, lse_s = -inf). Launch 2
 * merges the chunks of each (b, h) with the rescaling rule of P3 "Step 4":
 * m* = max_s lse_s, w_s = exp(lse_s - m*), o = sum_s w_s o_s / sum_s w_s,
 * lse = m* + log(sum_s w_s).
 *
 *   q            device BF16 [B,H,1,d].
 *   k, v         device BF16 [B,H,Nk,d].
 *   o            device BF16 [B,H,1,d] (written).
 *   lse          device FP32 [B,H,1] (written); may be NULL.
 *   B, H, Nk, d  sizes (d in {64,128}); Nk >= 0.
 *   scale        score scale; finite and > 0.
 *   seqlens_k    device int32 [B] of visible key counts, or NULL for Nk.
 *   num_splits   1 <= num_splits <= 1024.
 *   workspace    device scratch of at least
 *                attn_decode_workspace_bytes(B, H, d, num_splits) bytes,
 *                256-byte aligned, owned by the caller; its contents are
 *                overwritten. Two calls that share one workspace must be
 *                ordered on the same stream.
 *   workspace_bytes  its size.
 *   stream       CUDA stream.
 */
attn_status_t attn_decode_splitkv(const void* q, const void* k, const void* v,
                                  void* o, float* lse,
                                  int B, int H, int Nk, int d, float scale,
                                  const int* seqlens_k, int num_splits,
                                  void* workspace, size_t workspace_bytes,
                                  attn_stream_t stream);

/*
 * attn_decode_splitkv_noalloc -- attn_decode_splitkv for callers that cannot
 * allocate device memory on their call path (for example a serving process
 * whose device memory is all reserved for its own pool, or one that must not
 * call cudaMalloc/cudaFree there because those calls can synchronise the
 * device). The source pages have no counterpart to this entry point: it only
 * changes where the per-split partials are kept.
 *
 * Same arguments, layout and result as attn_decode_splitkv, without the
 * workspace: the partials go to a fixed 4 MiB array inside the library
 * (allocated by the CUDA loader, held on every GPU that loads the library
 * until the process exits). The call allocates nothing.
 *   - Limit: attn_decode_workspace_bytes(B, H, d, num_splits) must be at most
 *     4 MiB (4194304 bytes); larger problems return ATTN_ERR_INVALID_ARG with
 *     a message, and need attn_decode_splitkv with a caller workspace.
 *   - The first call on a device looks up the array's device address on
 *     that device (cudaGetSymbolAddress); make that first call before any
 *     stream capture.
 *   - Every call on a device shares the one array, which keeps the last
 *     call's contents (no part of it needs to start at zero). Calls whose
 *     kernels overlap on the GPU, e.g. on two unordered streams, race on it:
 *     order them on one stream.
 */
attn_status_t attn_decode_splitkv_noalloc(const void* q, const void* k, const void* v,
                                          void* o, float* lse,
                                          int B, int H, int Nk, int d, float scale,
                                          const int* seqlens_k, int num_splits,
                                          attn_stream_t stream);

/*
 * attn_softmax_rows -- row softmax y = softmax(x) of a [rows, n] matrix with
 * the online normalizer (P3 "Online softmax": "Step 2" keeps the pair
 * (m, l) -- running maximum and sum of exp(x - m), the sum rescaled by
 * exp(m_old - m_new) when the maximum grows -- in one pass; "Step 3" writes
 * exp(x_i - m) / l in a second pass; "Step 4" merges the pairs of the
 * threads that share a row, in any grouping).
 *
 *   x, y     device pointers, [rows, n] row-major, same dtype (ATTN_DTYPE_F32
 *            or ATTN_DTYPE_BF16), aligned to the element size (16-byte
 *            aligned rows with n a multiple of 16 bytes take the vector path).
 *            x and y may be the same buffer.
 *   lse      device FP32 [rows] (written: m + log l, natural log), or NULL.
 *   rows     0 <= rows < 2^31; n >= 1.
 * Entries may be -inf (weight 0); a row of only -inf gives y = 0 and
 * lse = -inf. Arithmetic is FP32; BF16 outputs are rounded once.
 */
attn_status_t attn_softmax_rows(const void* x, void* y, float* lse, long long rows, int n,
                                int dtype, attn_stream_t stream);

/*
 * attn_check_device_error -- synchronise `stream`, then report whether any
 * kernel of this library on the current device gave up a bounded wait since
 * the last call (ATTN_ERR_TIMEOUT, and the error word is cleared), or
 * whether the stream itself reported a CUDA error (ATTN_ERR_CUDA).
 */
attn_status_t attn_check_device_error(attn_stream_t stream);

/*
 * attn_exp2_soft -- diagnostic: y[i] = 2^x[i] by the software exponential
 * the forward kernels use for part of the attention weights (the partial
 * move of exponentials from the special-function unit to the FMA units that
 * P1, "What did FlashAttention-2 and -3 change?", attributes to
 * FlashAttention-4): Cody-Waite reduction n = round(x), f = x - n, then a
 * degree-3 minimax polynomial for 2^f (relative error <= 1.02e-4 for
 * -126 <= x <= 127) and n added to the exponent. x <= -127 (and -inf)
 * gives +0; -127 < x < -126 gives a denormal below 2^-126.
 *   x, y    device FP32 [n], 4-byte aligned; n >= 0. Asynchronous on stream.
 */
attn_status_t attn_exp2_soft(const float* x, float* y, long long n, attn_stream_t stream);

/*
 * attn_selftest_bounded_wait -- diagnostic: launch one CTA that waits on a
 * shared-memory barrier that nothing ever completes, with a limit of
 * `limit_cycles` SM clock cycles (1 .. 2^31). The wait must give up, record
 * the timeout in the error word and return, so that the following
 * attn_check_device_error() reports ATTN_ERR_TIMEOUT and the context stays
 * usable. Used by the tests of the failure path; faults nothing.
 */
attn_status_t attn_selftest_bounded_wait(long long limit_cycles,
                                         attn_stream_t stream);

/* attn_last_error -- message of the last failed call on this host thread
 * ("" if none). The pointer stays valid until the next call on the thread. */
const char* attn_last_error(void);

/* attn_version -- library version string. */
const char* attn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_H_ */
