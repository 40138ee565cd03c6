/*
 * attn.h -- C ABI of the GB300 (sm_103a) multi-head scaled dot-product
 * attention forward library (libattn_gb300.so).
 *
 * The operation (eq. (1) of "Attention Is All You Need", section 3.2.1, as
 * restated on every page read for this library; the masks of section 3.2.3):
 *
 *     O[b,h] = softmax(Q[b,h] K[b,h]^T * scale + M) V[b,h]
 *     LSE[b,h,i] = ln sum_j exp(scale * q_i.k_j + M_ij)
 *
 * for every batch entry b and head h, with M_ij = -inf on forbidden
 * connections and 0 elsewhere:
 *   ATTN_MASK_NONE         encoder self-attention: every query sees every key;
 *   ATTN_MASK_CAUSAL       decoder masked self-attention: query i sees keys
 *                          j <= i (itself included), top-left aligned when
 *                          n_q != n_k;
 *   ATTN_MASK_KEY_PADDING  encoder-decoder attention over padded sequences:
 *                          query rows of batch entry b see keys j < key_lens[b].
 * A query row with no visible key gets O = 0 and LSE = -inf.  The usual
 * scale is 1/sqrt(d_k); it is an argument so that the caller states it.
 *
 * Layout (all entry points): contiguous [B, h, n, d] tensors, d innermost;
 * Q [B,h,n_q,d_k], K [B,h,n_k,d_k], V [B,h,n_k,d_v], O [B,h,n_q,d_v] with
 * d_v = d_k, LSE [B,h,n_q] float32.
 *
 * Ownership and execution: every pointer argument is a device pointer owned
 * by the caller; the library reads its inputs and writes only the outputs
 * (and workspace) each call names, never frees caller memory, and allocates
 * no device memory.  Calls
 * are asynchronous on `stream` (NULL = the legacy default stream): argument
 * checks happen on the host before anything is enqueued; errors found on the
 * device are reported by attn_check().  No call synchronises the host.
 * Errors are returned as attn_status codes; nothing is thrown across the ABI.
 */
#ifndef ATTN_GB300_H_
#define ATTN_GB300_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st; /* cudaStream_t */

typedef enum {
  ATTN_MASK_NONE = 0,
  ATTN_MASK_CAUSAL = 1,
  ATTN_MASK_KEY_PADDING = 2,
  ATTN_MASK_WINDOW = 3 /* attn_fwd_strided only: the window of attn_fwd_window */
} attn_mask_kind;

typedef enum {
  ATTN_OK = 0,
  ATTN_ERR_INVALID_ARG = -1, /* null/misaligned pointer, size < 1, bad mask or scale */
  ATTN_ERR_UNSUPPORTED = -2, /* head size or device the library does not cover */
  ATTN_ERR_CUDA = -3,        /* a CUDA runtime/driver call failed, see attn_last_cuda_error */
  ATTN_ERR_TIMEOUT = -4,     /* a kernel gave up on a bounded wait (see attn_check) */
  ATTN_ERR_SCRATCH_TOO_SMALL = -5 /* attn_decode_noalloc: sizes need more than its fixed scratch */
} attn_status;

/*
 * attn_fwd -- bf16 forward on the tensor cores (tcgen05 + TMEM + TMA).
 *   q, k, v : const __nv_bfloat16*, layout above, 16-byte aligned.
 *   o       : __nv_bfloat16* [B,h,n_q,d_k], written (rounded to nearest even).
 *   lse     : float* [B,h,n_q] or NULL (then not written).
 *   B, h, n_q, n_k >= 1; d_k in {16, 32, 64, 128} (the head sizes of the
 *             model variants of "Attention Is All You Need", Table 3, rows (A)
 *             and (B), that fit the tensor-core path; others:
 *             ATTN_ERR_UNSUPPORTED).
 *   scale   : finite and > 0 (normally 1/sqrt(d_k)).
 *   mask_kind : an attn_mask_kind.
 *   key_lens  : device int32[B], required for ATTN_MASK_KEY_PADDING, ignored
 *               otherwise; values are clamped to [0, n_k] on the device.
 *   stream  : cudaStream_t.
 * Scores, softmax and the P.V product are computed in fp32 from bf16 inputs;
 * P is rounded to bf16 before the second product.  K and V rows past
 * key_lens[b] never affect the result but must hold finite values: the
 * tensor-core product multiplies the tail of a partly valid tile by zero.
 */
int attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int h,
             int n_q, int n_k, int d_k, float scale, int mask_kind, const int* key_lens,
             struct CUstream_st* stream);

/*
 * attn_fwd_window -- attn_fwd with restricted self-attention: query i sees
 * the keys j with  i - window_left <= j <= i + window_right  (and j < n_k),
 * every other connection is -inf before the softmax.  window_left =
 * window_right = w gives the neighbourhood of 2w + 1 positions centred on
 * the output position that "Attention Is All You Need" proposes for very
 * long sequences (section 4 and Table 1: O(r n d) work instead of O(n^2 d));
 * window_right = 0 gives a causal window of window_left + 1 positions.
 * Tiles outside every row's window are never loaded.  Arguments otherwise as
 * attn_fwd (bf16, d_k in {16, 32, 64, 128}); window_left, window_right >= 0
 * (ATTN_ERR_INVALID_ARG otherwise).  A query whose window holds no key
 * (i - window_left >= n_k) gets O = 0, LSE = -inf.
 */
int attn_fwd_window(const void* q, const void* k, const void* v, void* o, float* lse, int B, int h,
                    int n_q, int n_k, int d_k, float scale, int window_left, int window_right,
                    struct CUstream_st* stream);

/*
 * attn_fwd_strided -- attn_fwd on tensors of any row, head and batch strides,
 * e.g. [B, n, h, d] (the layout a projection to h heads produces) or Q, K, V
 * packed in one [B, n, 3, h, d] buffer, without a copy.  Element (b, hh, i, t)
 * of Q is  q[b*q_strides[0] + hh*q_strides[1] + i*q_strides[2] + t], and the
 * same for k, v and o (o is written through its strides; lse stays
 * contiguous [B, h, n_q]).  Strides are host arrays of 3 element counts, each
 * > 0 and a multiple of 8 (16 bytes); d is contiguous.  mask_kind: any
 * attn_mask_kind; ATTN_MASK_WINDOW uses window_left / window_right as
 * attn_fwd_window does (both ignored otherwise).  bf16, d_k in {16, 32, 64,
 * 128}; the tensors must not overlap o.  Other arguments as attn_fwd.
 */
int attn_fwd_strided(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                     int h, int n_q, int n_k, int d_k, const int64_t* q_strides,
                     const int64_t* k_strides, const int64_t* v_strides, const int64_t* o_strides,
                     float scale, int mask_kind, const int* key_lens, int window_left,
                     int window_right, struct CUstream_st* stream);

/*
 * attn_fwd_host -- attn_fwd (any mask_kind, as attn_fwd_strided) on HOST
 * buffers: q, k, v are copied to the device, the forward runs there, and o
 * (and lse, if not NULL) are copied back, all enqueued on `stream` without a
 * host synchronisation.  The batch is cut into up to 8 slices of whole batch
 * entries whose copies in, forward and copies out are pipelined over two
 * internal copy streams (one each way), so the copies of one slice overlap
 * the others' work;
 * each (b, h) is computed by the same kernel as attn_fwd, so o and lse are
 * bitwise those of attn_fwd.  Work enqueued on `stream` before the call
 * completes before the first copy starts, and work enqueued after it waits
 * for the last copy.
 *   q, k, v, o : host bf16 [B, h, n, d_k] (contiguous); lse: host float
 *              [B, h, n_q] or NULL; key_lens: host int32[B] for
 *              ATTN_MASK_KEY_PADDING.  Pinned (page-locked) host memory lets
 *              the copies run asynchronously; pageable memory is correct but
 *              slower.  The host buffers must stay valid until the stream
 *              reaches the end of the call's work.
 *   dev_buf, dev_buf_bytes : caller-owned device staging of at least
 *              attn_fwd_host_buffer_bytes(B, h, n_q, n_k, d_k) bytes,
 *              256-byte aligned; overwritten.
 * Other arguments and status codes as attn_fwd_strided (bf16, d_k in {16, 32,
 * 64, 128}).
 */
int attn_fwd_host(const void* q, const void* k, const void* v, void* o, float* lse, int B, int h,
                  int n_q, int n_k, int d_k, float scale, int mask_kind, const int* key_lens,
                  int window_left, int window_right, void* dev_buf, size_t dev_buf_bytes,
                  struct CUstream_st* stream);

/* Device staging bytes attn_fwd_host needs for these sizes (0 for unsupported sizes). */
size_t attn_fwd_host_buffer_bytes(int B, int h, int n_q, int n_k, int d_k);

/*
 * attn_fwd_f32 -- float32 forward on the CUDA cores (fp32 FMA, same
 * definition, same arguments with float tensors).  d_k in {16, 32, 64, 128}.
 */
int attn_fwd_f32(const float* q, const float* k, const float* v, float* o, float* lse, int B,
                 int h, int n_q, int n_k, int d_k, float scale, int mask_kind,
                 const int* key_lens, struct CUstream_st* stream);

/*
 * attn_decode -- the same operation for a few new queries against a
 * key/value cache (an autoregressive decoding step): query i of (b, h) sees
 * the cached keys j < cache_lens[b].  Bound by HBM bandwidth; runs on the
 * CUDA cores with TMA-fed tiles and splits each head's cache across CTAs when
 * B*h alone would leave SMs idle.
 *   q        : bf16 [B, h, n_q, d_k], 1 <= n_q <= 8.
 *   k_cache, v_cache : bf16 [B, h, L_max, d_k]; rows past cache_lens[b] are
 *              never used.
 *   o, lse   : bf16 [B, h, n_q, d_k] and float [B, h, n_q] (lse may be NULL).
 *   d_k      : 16, 32, 64 or 128 (else ATTN_ERR_UNSUPPORTED; 64 runs the TMA-fed
 *              kernel, the others a kernel with plain loads); B*h <= 65535.
 *   cache_lens : device int32[B] (clamped to [0, L_max] on the device), or
 *              NULL when every sequence fills the cache.
 *   workspace, workspace_bytes : caller-owned device scratch of at least
 *              attn_decode_workspace_bytes(...) bytes (16-byte aligned) for the
 *              per-chunk partial results; may be NULL when that size is 0.
 */
int attn_decode(const void* q, const void* k_cache, const void* v_cache, void* o, float* lse,
                int B, int h, int n_q, int L_max, int d_k, float scale, const int* cache_lens,
                void* workspace, size_t workspace_bytes, struct CUstream_st* stream);

/* Scratch bytes attn_decode needs for these sizes on the current device
 * (0 when no split is needed, or for unsupported sizes). */
size_t attn_decode_workspace_bytes(int B, int h, int n_q, int L_max, int d_k);

/*
 * attn_decode_strided -- attn_decode on a query, a cache and an output of any
 * batch, head and row strides, e.g. a cache laid out [B, L_max, h, d] as many
 * decoders keep it.  Element (b, hh, i, t) of each tensor X is
 * x[b*s[0] + hh*s[1] + i*s[2] + t]; strides is a host array of 12 element
 * counts, three (b, h, row) per tensor in the order q, k_cache, v_cache, o,
 * each > 0 and a multiple of 8 (16 bytes); d is contiguous; lse stays
 * contiguous [B, h, n_q].  Other arguments, the workspace size and the status
 * codes as attn_decode.
 */
int attn_decode_strided(const void* q, const void* k_cache, const void* v_cache, void* o,
                        float* lse, int B, int h, int n_q, int L_max, int d_k,
                        const int64_t* strides, float scale, const int* cache_lens,
                        void* workspace, size_t workspace_bytes, struct CUstream_st* stream);

/*
 * attn_decode_window -- attn_decode with restricted self-attention
 * ("Attention Is All You Need", section 4 and Table 1: each output position
 * attends only to a neighbourhood of r positions around itself).  In a
 * decoder the neighbourhood of the newest position holds only that position
 * and earlier ones, so every query of (b, h) sees the cached keys j with
 *   cache_lens[b] - 1 - window <= j < cache_lens[b]
 * (the newest cached key and the `window` keys before it; attn_fwd_window
 * with window_right = 0 at the last position).  Keys before the window are
 * never read.  window >= 0 (ATTN_ERR_INVALID_ARG otherwise); a window of at
 * least L_max - 1 gives attn_decode's result.  workspace_bytes must be at
 * least attn_decode_window_workspace_bytes(B, h, n_q, L_max, d_k, window)
 * (the cache is split by the window's length, not by L_max).  Other
 * arguments, layouts and status codes as attn_decode.
 */
int attn_decode_window(const void* q, const void* k_cache, const void* v_cache, void* o,
                       float* lse, int B, int h, int n_q, int L_max, int d_k, float scale,
                       const int* cache_lens, int window, void* workspace,
                       size_t workspace_bytes, struct CUstream_st* stream);

/* Scratch bytes attn_decode_window needs (0 when no split is needed, for
 * unsupported sizes or for window < 0). */
size_t attn_decode_window_workspace_bytes(int B, int h, int n_q, int L_max, int d_k, int window);

/* Size of the fixed scratch array behind attn_decode_noalloc (1 MiB). */
#define ATTN_DECODE_NOALLOC_SCRATCH_BYTES (1u << 20)

/*
 * attn_decode_noalloc -- attn_decode without the workspace argument, for
 * callers that cannot allocate device memory on the call path: an engine
 * that plans all of its device memory ahead and allows no allocation while
 * it serves requests, a plug-in that is handed only its input and output
 * buffers, or a caller for whom the device-wide synchronisation an
 * allocation may cause is not acceptable.  (This entry point has no
 * counterpart in the paper; it only changes where the scratch lives.)
 *
 * The per-chunk partial results go to an array of
 * ATTN_DECODE_NOALLOC_SCRATCH_BYTES that the library declares in its own
 * device memory: every device that loads the library holds it until the
 * process exits, and nothing is allocated or freed per call.  Sizes whose
 * partials would not fit return ATTN_ERR_SCRATCH_TOO_SMALL (use attn_decode
 * with a workspace of attn_decode_workspace_bytes(...) instead).
 *
 * The first call on a device whose sizes split the cache (the calls for
 * which attn_decode_workspace_bytes is not 0; only those use the array)
 * looks up the array's device address, once per device, with that device
 * current; make such a call before any stream capture.  All calls share the one array and it keeps whatever the last call
 * left in it; nothing in it needs to start at zero (every partial is written
 * before it is read).  Calls whose kernels may overlap on the GPU (different
 * streams, or host threads on the same device) race on the array: order them
 * on one stream.  Arguments and results otherwise as attn_decode.
 */
int attn_decode_noalloc(const void* q, const void* k_cache, const void* v_cache, void* o,
                        float* lse, int B, int h, int n_q, int L_max, int d_k, float scale,
                        const int* cache_lens, struct CUstream_st* stream);

/*
 * attn_bwd -- gradients of attn_fwd: given dout = dLoss/dO, writes
 *   dq = dLoss/dQ, dk = dLoss/dK, dv = dLoss/dV
 * for the same (q, k, v, scale, mask_kind, key_lens).  Per (b, h), with
 * P = softmax(scale * Q K^T + M) recomputed from q, k and lse:
 *   dV = P^T dO,  dP = dO V^T,  D_i = sum_c dO[i,c] O[i,c],
 *   dS = P * (dP - D_i),  dQ = scale dS K,  dK = scale dS^T Q.
 * This is the back-propagation through eq. (1) of "Attention Is All You
 * Need" (section 3.2.1) that training the model (section 5) needs; the
 * paper does not write it out.
 *   q, k, v  : bf16, as for attn_fwd; d_k = d_v in {16, 32, 64}, else
 *              ATTN_ERR_UNSUPPORTED (d_k = 128 is forward-only).
 *   o, lse   : the output and log-sum-exp attn_fwd returned for these inputs
 *              (lse is required here).
 *   dout     : bf16 [B, h, n_q, d_k].
 *   dq, dk, dv : bf16 outputs shaped like q, k, v (rounded to nearest even).
 *              Key rows past key_lens[b] (or that no query sees) get zeros.
 *   workspace, workspace_bytes : caller-owned device scratch of at least
 *              attn_bwd_workspace_bytes(B, h, n_q, d_k) bytes, 16-byte aligned
 *              (per-row softmax statistics and an fp32 dQ accumulator); its
 *              contents on entry do not matter.
 * Products run on the tensor cores from bf16 operands with fp32
 * accumulation; P and dS are rounded to bf16 before the products that use
 * them.  Three kernels are enqueued on `stream`.
 */
int attn_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout,
             const float* lse, void* dq, void* dk, void* dv, int B, int h, int n_q, int n_k,
             int d_k, float scale, int mask_kind, const int* key_lens, void* workspace,
             size_t workspace_bytes, struct CUstream_st* stream);

/*
 * attn_bwd_window -- the gradients of attn_fwd_window (restricted
 * self-attention: query i sees keys i - window_left .. i + window_right).
 * Arguments as attn_bwd with mask_kind and key_lens replaced by the window
 * sides (>= 0, else ATTN_ERR_INVALID_ARG); o and lse must come from
 * attn_fwd_window with the same window.  Keys no query's window reaches get
 * dk = dv = 0; queries whose window holds no key get dq = 0.
 */
int attn_bwd_window(const void* q, const void* k, const void* v, const void* o, const void* dout,
                    const float* lse, void* dq, void* dk, void* dv, int B, int h, int n_q,
                    int n_k, int d_k, float scale, int window_left, int window_right,
                    void* workspace, size_t workspace_bytes, struct CUstream_st* stream);

/*
 * attn_bwd_strided -- attn_bwd (or attn_bwd_window) on tensors of any row,
 * head and batch strides, the gradient of attn_fwd_strided: element
 * (b, hh, i, t) of each tensor X is  x[b*s[0] + hh*s[1] + i*s[2] + t].
 * strides is a host array of 24 element counts, three (b, h, row) per tensor
 * in the order q, k, v, o, dout, dq, dk, dv; each > 0 and a multiple of 8 (16
 * bytes); d is contiguous.  dq, dk, dv are written through their strides (for
 * instance into one packed [B, n, 3, h, d] gradient buffer) and must not
 * overlap the inputs; lse stays contiguous [B, h, n_q].  mask_kind: any
 * attn_mask_kind; ATTN_MASK_WINDOW uses window_left / window_right as
 * attn_bwd_window does (both ignored otherwise).  Other arguments as
 * attn_bwd (d_k in {16, 32, 64}; the same workspace size).
 */
int attn_bwd_strided(const void* q, const void* k, const void* v, const void* o, const void* dout,
                     const float* lse, void* dq, void* dk, void* dv, int B, int h, int n_q,
                     int n_k, int d_k, const int64_t* strides, float scale, int mask_kind,
                     const int* key_lens, int window_left, int window_right, void* workspace,
                     size_t workspace_bytes, struct CUstream_st* stream);

/* Scratch bytes attn_bwd needs for these sizes (0 for unsupported sizes). */
size_t attn_bwd_workspace_bytes(int B, int h, int n_q, int d_k);

/*
 * attn_check -- synchronise `stream`, then report (and clear) any error a
 * kernel of this library recorded on the current device since the last check:
 * ATTN_ERR_TIMEOUT when a bounded wait inside a kernel ran out (the kernel
 * returned early and its outputs are incomplete), ATTN_ERR_CUDA when the
 * synchronisation itself failed, else ATTN_OK.
 */
int attn_check(struct CUstream_st* stream);

/* Static description of a status code. */
const char* attn_status_string(int status);

/* The cudaError_t behind the most recent ATTN_ERR_CUDA in this process. */
int attn_last_cuda_error(void);

/*
 * attn_set_wait_limit_ns -- wall-clock limit for every bounded wait inside
 * the kernels launched after this call (default 2e9 ns).  0 restores the
 * default.  Returns the previous value.
 */
uint64_t attn_set_wait_limit_ns(uint64_t limit_ns);

/* Number of kernels this library has launched in this process. */
uint64_t attn_launch_count(void);

/* ------------------------------------------------------------------------
 * Diagnostics (not part of the attention operation; used by the tests).
 * ------------------------------------------------------------------------ */

/*
 * attn_diag_tile -- one CTA runs the two tensor-core products of a single
 * 128x128 tile exactly as the fused kernel issues them:
 *   s = q k^T  (q, k: bf16 [128, 64]; s: float [128, 128])
 *   o = p v    (p: bf16 [128, 128]; v: bf16 [128, 64]; o: float [128, 64])
 * q, k and v are staged by TMA with 128-byte swizzle, p is written to tensor
 * memory by the threads, both products accumulate in tensor memory and are
 * read back with tcgen05.ld.  All pointers are device pointers, 16-byte
 * aligned.
 */
int attn_diag_tile(const void* q, const void* k, const void* p, const void* v, float* s,
                   float* o, struct CUstream_st* stream);

/*
 * attn_diag_wait_timeout -- launch a one-thread kernel that waits on an
 * mbarrier nobody arrives on, bounded by `limit_ns`; it records
 * ATTN_ERR_TIMEOUT for attn_check() and returns.  Exercises the failure path
 * of the bounded waits without faulting the GPU.
 */
int attn_diag_wait_timeout(uint64_t limit_ns, struct CUstream_st* stream);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_GB300_H_ */
