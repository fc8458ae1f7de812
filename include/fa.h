/*
 * fa.h — exact softmax attention on GB300 (sm_103a): the C ABI.
 *
 * The library computes O = softmax(scale * Q K^T) V tile by tile with an online
 * softmax, so the N x N score matrix never reaches device memory, and stores one
 * logsumexp per query row; the backward pass recomputes the probabilities from
 * that logsumexp.  Sources, by page and section:
 *   - "FlashAttention" (deep dive, tirogla.com), section "How it works": inputs
 *     Q, K, V of shape N x d per head, outputs O and one logsumexp per row, no
 *     state between calls; L = m + log l; the backward pass recomputes
 *     P = exp(Q K^T * scale - L) and uses D = rowsum(dO o O), dS = P o (dP - D).
 *   - "tm_flash_attention_arch_2k", section "End-to-end forward pass": the
 *     [B, H, N, d] layout; section "The architecture: every step explained":
 *     causal blocks above the diagonal have no effect and are skipped.
 *   - "FlashAttention" (deep dive), section "Code" (the GPU kernel): tensors
 *     contiguous as (B*H, N, d), 64-bit offsets; section "Pitfalls": int32
 *     offset overflow, fully masked rows.
 *
 * Conventions shared by every entry point:
 *   - Layout: q, k, v, o, dO, dq, dk, dv are [B, H, N, d] contiguous (row stride
 *     d elements, head stride N*d); lse is [B, H, N] float32.  Queries and keys
 *     have the same length N.
 *   - Masking: causal != 0 applies the square, top-left aligned mask: key j is
 *     visible to query i iff j <= i.  causal == 0 attends to all N keys.
 *   - lse holds the natural-log logsumexp of the scaled scores over the visible
 *     keys: lse_i = log(sum_j exp(scale * q_i . k_j)).
 *   - Pointers are device pointers, 16-byte aligned (the tensor-memory-access
 *     engine needs it); lse 4-byte aligned.
 *   - Ownership: the caller allocates and owns every buffer, workspaces
 *     included.  The library allocates no device memory, keeps no state
 *     between calls (beyond per-device one-time set-up) and never synchronises
 *     the stream: work is enqueued on `stream` and the call returns.  Inputs
 *     are read only; outputs are fully overwritten.
 *   - Errors: every entry point returns an fa_status.  Argument errors are
 *     detected on the host before anything is enqueued.  A device-side wait
 *     that exceeds its time limit sets a device status word, read with
 *     fa_get_device_status().  No C++ exception and no exit() crosses this ABI.
 *   - Supported: head dim d in {64, 128}; N >= 1 of any value; B*H*N*d below
 *     2^62; compute capability 10.3 (GB300).
 */
#ifndef FA_GB300_H
#define FA_GB300_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st *fa_stream_t;

typedef enum fa_status {
    FA_OK = 0,
    FA_ERR_INVALID_ARG = 1,     /* NULL pointer, B/H/N < 1, H not a multiple of Hkv, non-finite scale, size overflow */
    FA_ERR_UNSUPPORTED = 2,     /* d not supported, or the device is not compute capability 10.3 */
    FA_ERR_ALIGNMENT = 3,       /* a pointer is not 16-byte aligned (lse: 4-byte) */
    FA_ERR_WORKSPACE = 4,       /* workspace NULL or smaller than fa_bwd_workspace_size() */
    FA_ERR_CUDA = 5,            /* a CUDA runtime/driver call failed; see fa_last_cuda_error() */
    FA_ERR_DEVICE_TIMEOUT = 6   /* a device-side wait gave up (read via fa_get_device_status) */
} fa_status;

/*
 * Forward pass, bf16 storage, fp32 accumulation.
 *   q, k, v  [B,H,N,d] bf16, read only
 *   o        [B,H,N,d] bf16, written: softmax(scale * q k^T [masked]) v
 *   lse      [B,H,N]   fp32, written: natural-log logsumexp per query row
 *   scale    multiplies the raw dot products (usually 1/sqrt(d)); must be finite
 * Page: "FlashAttention" (deep dive), section "How it works" (the forward loop
 * with running max m, running sum l and accumulator acc; O = acc / l and
 * L = m + log l are the only outputs).
 */
int fa_fwd(const void *q, const void *k, const void *v, void *o, float *lse,
           int B, int H, int N, int d, float scale, int causal, fa_stream_t stream);

/*
 * Grouped-query forward (GQA; multi-query attention when Hkv = 1): H query heads
 * share Hkv key/value heads, query head h reading key/value head h / (H / Hkv).
 *   q, o  [B,H,N,d] bf16;  k, v  [B,Hkv,N,d] bf16;  lse [B,H,N] fp32
 *   H must be a multiple of Hkv (else FA_ERR_INVALID_ARG).  fa_fwd is Hkv = H.
 * Page: "FlashAttention" (deep dive), section "Implementation notes" (several query
 * heads map to one key/value head; the loads are shared and nothing else changes).
 */
int fa_fwd_gqa(const void *q, const void *k, const void *v, void *o, float *lse,
               int B, int H, int Hkv, int N, int d, float scale, int causal, fa_stream_t stream);

/*
 * Forward pass with float32 inputs and outputs (same layout and meaning as
 * fa_fwd; q, k, v, o are float32).  The two products run on the tensor cores
 * in TF32 with fp32 accumulation.  Supported for d = 64 only (the fp32 workload:
 * one head, N = 256, d = 64, non-causal).
 * Page: "FlashAttention" (deep dive), section "How it works" (the same forward loop:
 * running max m and sum l, O = acc / l, L = m + log l) and its section "Code" (the
 * tiled loop on fp32 slices, one head, row-major N x d, checked against naive softmax
 * attention); tile sizes change only the summation order ("Flash Attention and
 * Memory-Efficient Attention Variants", active recall A3).
 */
int fa_fwd_f32(const float *q, const float *k, const float *v, float *o, float *lse,
               int B, int H, int N, int d, float scale, int causal, fa_stream_t stream);

/*
 * Bytes of device workspace fa_bwd needs for a problem of this size: the fp32
 * dQ accumulator plus two fp32 per-row vectors (D = rowsum(dO o O) and the
 * logsumexp in base 2), padded to whole 128-row tiles.  Returns 0 if the
 * arguments are invalid.
 * Page: "FlashAttention" (deep dive), section "How it works" (the backward pass
 * uses D = rowsum(dO o O) per query row and recomputes P from the saved L) and
 * section "Pitfalls" (dQ gathers contributions from every key block: summed across
 * thread blocks into one fp32 accumulator per element, which is this workspace).
 */
size_t fa_bwd_workspace_size(int B, int H, int N, int d);

/*
 * Backward pass, bf16 storage, fp32 accumulation.
 *   q, k, v, o  [B,H,N,d] bf16, read only (o and lse as written by fa_fwd)
 *   lse         [B,H,N]   fp32, read only
 *   dout        [B,H,N,d] bf16, read only: gradient of the loss w.r.t. o
 *   dq, dk, dv  [B,H,N,d] bf16, written: gradients w.r.t. q, k, v
 *   workspace   device buffer of at least fa_bwd_workspace_size(B,H,N,d)
 *               bytes, 256-byte aligned; its contents on entry do not matter
 *               and are scratch on exit
 * The dQ contributions of different key blocks are summed with fp32 bulk
 * reductions in an order that varies, so dq can differ from run to run in the last
 * bits; dk and dv are deterministic.  fa_bwd_deterministic gives bit-identical dq.
 * Page: "FlashAttention" (deep dive), section "How it works" (backward
 * recomputes P = exp(Q K^T * scale - L), D = rowsum(dO o O),
 * dS = P o (dP - D)); the scale enters dQ and dK by the chain rule.
 */
int fa_bwd(const void *q, const void *k, const void *v, const void *o, const float *lse,
           const void *dout, void *dq, void *dk, void *dv, void *workspace,
           size_t workspace_bytes, int B, int H, int N, int d, float scale, int causal,
           fa_stream_t stream);

/*
 * Grouped-query backward: as fa_bwd, with k, v, dk, dv [B,Hkv,N,d]; dk and dv sum
 * the contributions of all H / Hkv query heads that share each key/value head.
 * The workspace is fa_bwd_workspace_size(B, H, N, d) (per query head).
 */
int fa_bwd_gqa(const void *q, const void *k, const void *v, const void *o, const float *lse,
               const void *dout, void *dq, void *dk, void *dv, void *workspace,
               size_t workspace_bytes, int B, int H, int Hkv, int N, int d, float scale,
               int causal, fa_stream_t stream);

/*
 * Workspace bytes fa_bwd_deterministic needs for [B,H,N,d] queries (two fp32
 * vectors per query head, padded to whole 128-row tiles), or 0 if the arguments
 * are invalid.  Smaller than fa_bwd_workspace_size: there is no dQ accumulator.
 */
size_t fa_bwd_deterministic_workspace_size(int B, int H, int N, int d);

/*
 * Deterministic backward pass: the same gradients as fa_bwd_gqa (Hkv = H for plain
 * multi-head attention), bit-identical from run to run.  Each dQ row has a single
 * writer that sums the key blocks in a fixed order, so no reduction across thread
 * blocks is involved; dK and dV are computed per key block as in fa_bwd.  The
 * price is recomputing S and dP in the dQ pass (seven tile products per
 * query/key block pair instead of five).
 *   q, k, v, o, lse, dout, dq, dk, dv  as for fa_bwd_gqa
 *   workspace   device buffer of at least fa_bwd_deterministic_workspace_size(B,H,N,d)
 *               bytes, 256-byte aligned; scratch
 * Same status codes as fa_bwd.
 * Page: "FlashAttention" (deep dive), section "How it works" (the backward pass:
 * recompute P from the saved L, D = rowsum(dO o O), dS = P o (dP - D)); the pages do
 * not fix how dQ is summed across key blocks.
 */
int fa_bwd_deterministic(const void *q, const void *k, const void *v, const void *o,
                         const float *lse, const void *dout, void *dq, void *dk, void *dv,
                         void *workspace, size_t workspace_bytes, int B, int H, int Hkv,
                         int N, int d, float scale, int causal, fa_stream_t stream);

/*
 * Workspace bytes fa_decode needs (the chunks' partial triples), or 0 if the
 * arguments are invalid or unsupported.
 */
size_t fa_decode_workspace_size(int B, int H, int Hkv, int Nk, int d);

/*
 * Decoding: one query row per head against a long key/value sequence, the keys
 * split into chunks processed in parallel and merged.
 *   q          [B,H,d]       bf16, read only: the newest position's query per head
 *   k, v       [B,Hkv,Nk,d]  bf16, read only; Hkv divides H, H / Hkv <= 16; query
 *                            head h uses key/value head h / (H / Hkv)
 *   o          [B,H,d]       bf16, written: softmax(scale * q k^T) v (every key visible)
 *   lse        [B,H]         fp32, written: natural-log logsumexp of the scaled scores
 *   workspace  device buffer of at least fa_decode_workspace_size(B,H,Hkv,Nk,d)
 *              bytes, 256-byte aligned; scratch
 *   num_chunks chunks per key/value head: 0 lets the library choose (every CTA
 *              slot filled, the last wave of CTAs full), otherwise it is clamped to
 *              [1, min(ceil(Nk/64), 256)];
 *              chunks are whole multiples of 64 keys
 * d = 64 or 128.  Status codes as for fa_fwd; FA_ERR_UNSUPPORTED when H / Hkv > 16.
 * The result does not depend on num_chunks beyond fp32 rounding order.
 * Page: "FlashAttention" (deep dive), section "Implementation notes" (decoding with
 * one query row: parallelise over chunks of the keys and merge the partial
 * (m, l, acc) triples with the rescaling rule of the tiled forward pass).
 */
int fa_decode(const void *q, const void *k, const void *v, void *o, float *lse,
              void *workspace, size_t workspace_bytes, int B, int H, int Hkv, int Nk,
              int d, float scale, int num_chunks, fa_stream_t stream);

/*
 * FP8 forward with incoherent processing.  The pages give only the idea ("FlashAttention"
 * deep dive, section "How it works": fp8 with incoherent processing; "FlashAttention
 * Explained", section "Later versions": an FP8 low-precision mode); the reading taken:
 * e4m3 codes (round to nearest even, saturating at +-448) with one scale per
 * (batch, head); Q and K rows rotated by the same orthogonal diag(s) H / sqrt(d) (H the
 * Sylvester Hadamard matrix, s random signs drawn by the caller), which leaves Q K^T
 * unchanged and spreads outlier coordinates before rounding.
 */

/* Bytes of the transposed V codes for [B,H,N,d]: B*H*d*Npad, Npad = N rounded up to 16. */
size_t fa_fp8_v_bytes(int B, int H, int N, int d);

/*
 * Quantize Q or K for fa_fwd_fp8.
 *   x        [B,H,N,d] bf16, read only
 *   signs    d fp32 values of +-1 (device), or NULL for no rotation; use the same
 *            signs for Q and K.  With signs each row becomes (x o signs) H / sqrt(d),
 *            computed with the Walsh-Hadamard butterflies in fp32
 *   x8       [B,H,N,d] e4m3 codes, written
 *   descale  [B,H] fp32, written: amax / 448 of each (batch, head) slice (1/448 for an
 *            all-zero slice); codes = e4m3(x * (448 / amax))
 * d = 64 or 128.  Status codes as for fa_fwd.
 */
int fa_quantize_qk_fp8(const void *x, const float *signs, void *x8, float *descale, int B,
                       int H, int N, int d, fa_stream_t stream);

/*
 * Quantize V for fa_fwd_fp8: e4m3 codes with one scale per (batch, head), transposed
 *   v        [B,H,N,d] bf16, read only
 *   vt8      [B,H,d,Npad] e4m3 codes (keys contiguous; keys N..Npad-1 are zero codes),
 *            fa_fp8_v_bytes(B,H,N,d) bytes, written
 *   descale  [B,H] fp32, written as for fa_quantize_qk_fp8
 */
int fa_quantize_v_fp8(const void *v, void *vt8, float *descale, int B, int H, int N, int d,
                      fa_stream_t stream);

/*
 * FP8 forward: O = softmax(scale * (dq Q8)(dk K8)^T [causal]) (dv V8) with both products
 * on the tensor cores in e4m3 (P rounded to e4m3 before the second product; the row
 * sums stay in fp32).
 *   q8            [B,H,N,d] e4m3 codes, k8 [B,Hkv,N,d], vt8 [B,Hkv,d,Npad] (as written by
 *                 the quantize calls above; Q and K rotated alike or not at all)
 *   descale_q     [B,H] fp32; descale_k, descale_v [B,Hkv] fp32
 *   o             [B,H,N,d] bf16, written;  lse [B,H,N] fp32 natural log, written
 * d = 128 only (FA_ERR_UNSUPPORTED otherwise); Hkv divides H.
 */
int fa_fwd_fp8(const void *q8, const void *k8, const void *vt8, const float *descale_q,
               const float *descale_k, const float *descale_v, void *o, float *lse, int B,
               int H, int Hkv, int N, int d, float scale, int causal, fa_stream_t stream);

/* Size in bytes of the scratch array built into the library for fa_bwd_noalloc. */
#define FA_NOALLOC_SCRATCH_BYTES ((size_t)64 << 20)

/*
 * Backward pass without a workspace argument, for callers that cannot allocate device
 * memory (a plugin handed only tensors by a framework that owns all device memory, a
 * loop that must not call cudaMalloc, a process with a fixed memory budget).  The pages
 * have no counterpart: this is a convenience of this library.
 *   Arguments, layouts and results are those of fa_bwd; the workspace is a device
 *   array of FA_NOALLOC_SCRATCH_BYTES inside the library (held by every GPU that loads
 *   the library until the process exits).
 *   Returns FA_ERR_WORKSPACE when fa_bwd_workspace_size(B, H, N, d) exceeds
 *   FA_NOALLOC_SCRATCH_BYTES (use fa_bwd with a caller-owned workspace instead);
 *   otherwise the same statuses as fa_bwd.
 *   The first call on a device looks up the array's device address (with that device
 *   current); make that first call before any stream capture.  All calls share the
 *   array, so calls whose kernels overlap on the GPU (e.g. on two streams) race.
 *   `stream` must belong to the current device: the array used is the current
 *   device's, and a stream of another device is rejected with FA_ERR_INVALID_ARG.
 *   Allocates nothing: no cudaMalloc, cudaFree or allocating library routine.
 */
int fa_bwd_noalloc(const void *q, const void *k, const void *v, const void *o, const float *lse,
                   const void *dout, void *dq, void *dk, void *dv, int B, int H, int N, int d,
                   float scale, int causal, fa_stream_t stream);

/*
 * Bytes of device buffer fa_fwd_bwd_host needs: three slots, each holding one chunk
 * of chunk_heads heads (q, k, v, dout, o, dq, dk, dv in bf16, lse in fp32, and the
 * chunk's fa_bwd workspace), each part 256-byte aligned.  chunk_heads <= 0 picks
 * ceil(B*H / 16); a value above B*H is clamped to B*H.  Returns 0 if the arguments
 * are invalid.
 */
size_t fa_fwd_bwd_host_buffer_size(int B, int H, int N, int d, int chunk_heads);

/*
 * One training step of attention, forward then backward, on tensors in HOST memory:
 * the same results as fa_fwd followed by fa_bwd on device copies of the inputs, with
 * the host<->device copies overlapped with the kernels.  Every (batch, head) pair is
 * an independent problem ("FlashAttention" deep dive, section "How it works": the
 * inputs and outputs of one head, no state between calls), so the B*H heads are cut
 * into chunks of chunk_heads consecutive heads; chunk c is copied in on an internal
 * stream, computed on `stream` (even chunks) or an internal compute stream (odd
 * chunks), and copied out on another internal stream, while chunks c - 1 and c + 1
 * are being copied.  Within a chunk the forward starts once q, k and v have landed
 * (dout follows them), and o and lse are copied out once the forward is done, ahead
 * of dq, dk and dv.
 *   q, k, v, dout   [B,H,N,d] bf16, HOST memory, read only
 *   o, dq, dk, dv   [B,H,N,d] bf16, HOST memory, written
 *   lse             [B,H,N]   fp32, HOST memory, written
 *   dev_buf         device buffer of at least fa_fwd_bwd_host_buffer_size(B, H, N, d,
 *                   chunk_heads) bytes, 256-byte aligned, owned by the caller; scratch
 * Host buffers should be page-locked (cudaHostAlloc or cudaHostRegister): copies from
 * pageable memory are correct but do not overlap.  The call enqueues the work and
 * returns; the results are in host memory once `stream` reaches the point of the
 * call (synchronise `stream`).  Work enqueued earlier on `stream` happens before the
 * first copy.  The library creates three streams and a few events per device on
 * first use and reuses them; concurrent calls on one device are serialised while
 * they enqueue, and must use distinct buffers.
 * Returns the statuses of fa_fwd and fa_bwd (argument errors before anything is
 * enqueued; FA_ERR_WORKSPACE if dev_buf is NULL or too small, FA_ERR_ALIGNMENT if it
 * is not 256-byte aligned).  After a CUDA error part of the step may have been
 * enqueued and the outputs are undefined.
 */
int fa_fwd_bwd_host(const void *q, const void *k, const void *v, const void *dout, void *o,
                    float *lse, void *dq, void *dk, void *dv, void *dev_buf, size_t dev_buf_bytes,
                    int B, int H, int N, int d, float scale, int causal, int chunk_heads,
                    fa_stream_t stream);

/*
 * Error reporting.  The pages fix no error convention ("FlashAttention" deep dive,
 * section "Pitfalls", lists what to guard against: fully masked rows, 32-bit offset
 * overflow, head dims the tensor cores cannot take); the status codes above and the
 * three calls below are this library's own.
 *
 * Synchronises `stream`, then returns and clears the device status word of
 * the current device: FA_OK, or FA_ERR_DEVICE_TIMEOUT if a kernel gave up
 * waiting since the last call (its outputs are then undefined).  Returns
 * FA_ERR_CUDA if the synchronisation itself failed.
 */
int fa_get_device_status(fa_stream_t stream);

/*
 * Failure-detection self-test: enqueues a one-warp kernel on `stream` whose mbarrier
 * wait nothing ever satisfies.  After the wait's time limit (about one second) the
 * kernel records FA_ERR_DEVICE_TIMEOUT in the device status word and returns; the CUDA
 * context stays usable.  Read the result with fa_get_device_status().  Does no other
 * work.  The pages have no counterpart: this checks the library's own bounded waits.
 */
int fa_selftest_wait_timeout(fa_stream_t stream);

/* Static, human-readable name of a status code (never NULL).  The pages define no
 * error convention: the names are this library's own. */
const char *fa_status_string(int status);

/* The cudaError_t of the last call that returned FA_ERR_CUDA in this thread (the
 * pages define no error convention: this library's own). */
int fa_last_cuda_error(void);

#ifdef __cplusplus
}
#endif

#endif /* FA_GB300_H */
