/*
 * attn.h -- C ABI of the GB300 (sm_103a) masked scaled dot-product attention library.
 *
 * The library computes, for every batch b, head h and query row i,
 *
 *     out[b,h,i,:] = softmax_j( scale * Q[b,h,i,:] . K[b,h,j,:] + M[b,i,j] ) V[b,h,j,:]
 *
 * which is the attention equation of "Paper Deep Reading: Attention Is All
 * You Need", §04 Attention mechanics (softmax(Q K^T / sqrt(d_k) + M) V), run
 * for every head of multi-head attention at once (the head_i terms of the
 * same section's MultiHead equation, and the slide deck's "Multi-Head
 * Attention" slide).  The additive mask M is 0 where attention is allowed and
 * -inf where it is not:
 *   - ATTN_MASK_KEY_PADDING: key j of batch b is masked iff j >= key_lengths[b]
 *     ("the encoder mainly masks padding", §04);
 *   - ATTN_MASK_CAUSAL: key j is masked for query i iff j > i (the decoder's
 *     masked self-attention; §03 "Decoder layer" sets illegal future
 *     connections to -inf before the softmax);
 *   - both flags together: the union of both masked sets.
 * A query row with no allowed key is written as 0.
 *
 * The three uses named on the slide deck ("Three Applications of Attention")
 * map to: encoder self-attention (m == n, key padding), decoder
 * self-attention (m == n, causal) and encoder-decoder attention (m queries
 * from the decoder, n keys/values from the encoder, key padding).
 *
 * Layout: Q is [B][h][m][d_k], K and V are [B][h][n][d_k], out is
 * [B][h][m][d_k], all dense row-major with d_k fastest (d_v == d_k), in
 * device memory of the current CUDA device.  key_lengths is int32 [B] in
 * device memory.
 *
 * Ownership: the caller allocates and owns every buffer.  The library keeps
 * no per-call state and allocates no device memory; the only global state is
 * a small device status word that records a kernel giving up a bounded wait,
 * and the streams and events attn_fwd_host makes once per device.
 * attn_fwd_ws additionally takes a caller-owned workspace (see there).
 *
 * Asynchrony: every compute entry point only enqueues work on the given
 * stream (a cudaStream_t; NULL is the legacy default stream) and returns.  A
 * status other than ATTN_OK means nothing was enqueued.  Buffers must stay
 * valid until the stream has executed the work.  `out` must not overlap Q, K,
 * V or key_lengths.  Calls that overlap on the GPU may share inputs freely.
 *
 * Errors are reported through the return value; no function aborts, prints
 * or throws.
 */
#ifndef ATTN_GB300_ATTN_H
#define ATTN_GB300_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    ATTN_OK = 0,
    ATTN_ERR_NULL = 1,           /* a required pointer is NULL */
    ATTN_ERR_SHAPE = 2,          /* B, h, m, n out of range, or causal with m != n */
    ATTN_ERR_DTYPE = 3,          /* unknown dtype, or d_k not supported for that dtype */
    ATTN_ERR_MASK = 4,           /* mask_kind has bits other than KEY_PADDING | CAUSAL */
    ATTN_ERR_ALIGN = 5,          /* a tensor pointer is not 16-byte aligned */
    ATTN_ERR_UNSUPPORTED = 6,    /* the kernel asked for cannot run this call */
    ATTN_ERR_CUDA = 7,           /* a CUDA runtime call failed (device query, launch) */
    ATTN_ERR_DEVICE_TIMEOUT = 8, /* a kernel gave up a bounded wait (see attn_device_status) */
    ATTN_ERR_VALUE = 9,          /* scale is negative (other than ATTN_SCALE_DEFAULT) or not finite */
    ATTN_ERR_ALIAS = 10,         /* out overlaps Q, K, V or key_lengths */
    ATTN_ERR_SCRATCH = 11        /* the call needs more scratch than attn_fwd_noalloc holds */
} attn_status;

typedef enum {
    ATTN_MASK_NONE = 0,
    ATTN_MASK_KEY_PADDING = 1,
    ATTN_MASK_CAUSAL = 2,
    ATTN_MASK_WINDOW = 4 /* restricted self-attention; attn_fwd_window only */
} attn_mask_kind; /* bit flags: 3 = key padding and causal */

/*
 * Passing ATTN_SCALE_DEFAULT as `scale` asks the library for the formula's own
 * scale, 1/sqrt(d_k) ("Paper Deep Reading", §04: the dot products are divided by
 * sqrt(d_k) so that their variance stays near 1), computed on the host in double
 * and rounded to float.  Any other negative or non-finite scale is rejected.
 */
#define ATTN_SCALE_DEFAULT (-1.0f)

typedef enum {
    ATTN_BF16 = 0, /* bf16 in and out; fp32 accumulation and softmax state */
    ATTN_FP32 = 1  /* fp32 in and out; fp32 arithmetic throughout (no TF32) */
} attn_dtype;

typedef enum {
    ATTN_KERNEL_AUTO = 0,  /* let the library choose (what attn_fwd does) */
    ATTN_KERNEL_FLASH = 1, /* tcgen05/TMA flash kernel, 256 query rows per CTA tile (bf16, d_k a multiple of 8, <= 64) */
    ATTN_KERNEL_SHORT = 2, /* same machinery, two heads per CTA tile, whole head resident (bf16, d_k as FLASH, m <= 128) */
    ATTN_KERNEL_SIMT = 3,  /* CUDA-core fp32 kernel (fp32 or bf16, d_k <= 128) */
    ATTN_KERNEL_WIDE = 4,  /* tcgen05/TMA kernel for d_k == 128 (bf16): two 128-row query tiles of one
                              head per CTA, or two heads per CTA when m <= 128 and n <= 128 */
    ATTN_KERNEL_RESIDENT = 5 /* tcgen05/TMA kernel for short key sequences: one 128-row query tile of
                                one head per CTA with its Q, K and V resident, exact two-pass softmax
                                per row (bf16, d_k as FLASH, n <= 256, any m) */
} attn_kernel;

typedef struct {
    int32_t B;     /* batch size, >= 1 */
    int32_t h;     /* heads, >= 1 */
    int32_t m;     /* query rows per (batch, head), >= 1 */
    int32_t n;     /* key/value rows per (batch, head), >= 1 */
    int32_t d_k;   /* head width (d_v == d_k), 1..128; tensor cores take bf16 heads of a
                      multiple of 8 up to 64, or of 128 */
    int32_t dtype; /* attn_dtype */
} attn_dims;

/*
 * Masked scaled dot-product attention over all heads (see the top of this
 * file for the formula, layout, ownership and asynchrony).
 *
 *   Q, K, V      device tensors, layout above, element type dims->dtype; 16-byte aligned
 *   key_lengths  device int32 [B], 4-byte aligned; read only when mask_kind has
 *                KEY_PADDING (may be NULL otherwise).  Values are clamped to [0, n]
 *                on the device.
 *   mask_kind    attn_mask_kind bits
 *   scale        multiplies Q K^T; 1/sqrt(d_k) in the formula.  Must be finite and >= 0,
 *                or ATTN_SCALE_DEFAULT for 1/sqrt(d_k).
 *   out          device tensor [B][h][m][d_k] of dims->dtype; 16-byte aligned
 *   dims         shapes and dtype (host pointer)
 *   stream       cudaStream_t to enqueue on (NULL = legacy default stream)
 *
 * Returns ATTN_OK once the work is enqueued.  Rejects (nothing enqueued):
 * NULL pointers (ATTN_ERR_NULL), non-positive sizes or causal with m != n or
 * sizes whose element counts overflow int64 (ATTN_ERR_SHAPE), unsupported
 * dtype/d_k (ATTN_ERR_DTYPE), unknown mask bits (ATTN_ERR_MASK), unaligned
 * pointers (ATTN_ERR_ALIGN), bad scale (ATTN_ERR_VALUE), `out` overlapping
 * an input (ATTN_ERR_ALIAS), CUDA failures (ATTN_ERR_CUDA).  Inputs must be
 * finite: non-finite values propagate through the arithmetic as IEEE rules
 * dictate.  Kernel choice: bf16 with d_k a multiple of 8 up to 64 runs on tensor
 * cores, narrower heads zero-padded to 64 inside the kernel (ATTN_KERNEL_RESIDENT
 * when n <= 256, ATTN_KERNEL_SHORT when m <= 128 and n > 256, else
 * ATTN_KERNEL_FLASH); bf16 with d_k == 128 on ATTN_KERNEL_WIDE (tensor cores);
 * everything else runs ATTN_KERNEL_SIMT.  The resident kernel is launched as a
 * programmatic dependent of the kernel before it on the stream: its launch and
 * set-up overlap that kernel's tail, and it reads and writes memory only after
 * that kernel has completed (stream order is kept).
 */
attn_status attn_fwd(const void *Q, const void *K, const void *V,
                     const int32_t *key_lengths, int mask_kind, float scale,
                     void *out, const attn_dims *dims, void *stream);

/*
 * attn_fwd with an explicit kernel choice (attn_kernel).  Same arguments,
 * rules and errors as attn_fwd; additionally returns ATTN_ERR_UNSUPPORTED when
 * the kernel asked for cannot run the call (for example ATTN_KERNEL_SHORT with
 * m > 128, or a tensor-core kernel with fp32).  Lets tests and benchmarks run
 * each kernel on the same inputs.
 */
attn_status attn_fwd_kernel(const void *Q, const void *K, const void *V,
                            const int32_t *key_lengths, int mask_kind, float scale,
                            void *out, const attn_dims *dims, void *stream,
                            int kernel);

/* Bytes of device workspace attn_fwd_ws needs (host only, no CUDA call). */
size_t attn_workspace_size(void);

/*
 * attn_fwd with a caller-owned device workspace of at least
 * attn_workspace_size() bytes, 16-byte aligned, not overlapping any tensor.
 * The tensor-core kernels use it for a dynamic tile schedule: CTAs claim
 * tiles from a counter in the workspace, so faster SMs take more tiles and
 * the last tiles finish closer together (the schedule of attn_fwd is
 * static).  Results are identical either way.
 *
 * Contract: the workspace must be zero-filled before its first use (for
 * example with cudaMemsetAsync); every call returns it to zero-filled when
 * its kernel finishes, also after a bounded wait gave up.  Calls that may
 * run at the same time on the GPU (different streams) must use different
 * workspaces; calls ordered on one stream may share one.
 *
 * Errors as attn_fwd, plus: workspace NULL (ATTN_ERR_NULL), too small
 * (ATTN_ERR_SHAPE), unaligned (ATTN_ERR_ALIGN), overlapping a tensor or, with
 * KEY_PADDING, key_lengths (ATTN_ERR_ALIAS).
 */
attn_status attn_fwd_ws(const void *Q, const void *K, const void *V,
                        const int32_t *key_lengths, int mask_kind, float scale,
                        void *out, const attn_dims *dims, void *stream,
                        void *workspace, size_t workspace_bytes);

/* Size of the device array attn_fwd_noalloc uses as its workspace. */
#define ATTN_NOALLOC_SCRATCH_BYTES 256

/*
 * attn_fwd_noalloc: attn_fwd_ws without a caller-supplied workspace, for
 * callers that cannot allocate device memory when they call.  No page of the
 * method has a counterpart for this entry point; it is library plumbing.
 *
 * Who needs it: code that must not call cudaMalloc (or a framework
 * allocator) on its hot path -- cudaMalloc can synchronise the whole device
 * and stall every stream, so serving loops and latency-critical code
 * allocate everything up front and never again -- and code that runs inside
 * a host framework that owns all device memory and offers no scratch buffer
 * to the library.  This entry point calls no cudaMalloc, cudaFree or other
 * allocating routine.
 *
 * Scratch: instead of a workspace it uses a statically allocated device
 * array of ATTN_NOALLOC_SCRATCH_BYTES bytes inside the library.  Every GPU
 * that loads the library holds that array until the process exits.  The
 * first call on a device looks up the array's device address with that
 * device current (one-time set-up); make that first call before any stream
 * capture on that device.  The address is kept for the life of the process
 * (a failed lookup is retried by the next call): calls after a device reset
 * (cudaDeviceReset, or a new primary context) are not supported.  Calls whose
 * kernel uses the array (bf16 heads of width up to 64) zero its counters on
 * `stream` before their kernel.  All calls on a device share the one array:
 * calls that may run at the same time on the GPU (different streams) race
 * on it and must not be made; calls ordered on one stream are safe.
 *
 * Arguments, rules and errors as attn_fwd.  A call whose scratch need
 * (attn_workspace_size()) exceeds ATTN_NOALLOC_SCRATCH_BYTES is rejected
 * with ATTN_ERR_SCRATCH; ATTN_ERR_CUDA if the one-time address lookup or the
 * zeroing fails.
 */
attn_status attn_fwd_noalloc(const void *Q, const void *K, const void *V,
                             const int32_t *key_lengths, int mask_kind, float scale,
                             void *out, const attn_dims *dims, void *stream);

/* Bytes of device workspace attn_fwd_host needs for `dims` (host only, no CUDA
 * call): room for Q, K, V and out on the device, the key lengths and the tile
 * counters.  0 when dims is NULL or invalid. */
size_t attn_fwd_host_workspace_size(const attn_dims *dims);

/*
 * attn_fwd on HOST buffers: the same operation (the attention equation of
 * "Paper Deep Reading: Attention Is All You Need", §04, with the mask M), with Q, K, V,
 * key_lengths (int32 [B]) and out in host memory, laid out as for attn_fwd.
 * The call copies the inputs to the device, runs the kernels and copies the
 * output back, overlapping the three: the problem is cut into chunks of whole
 * (batch, head) slices (whole batches, or a range of heads of one batch);
 * chunk c's kernel starts as soon as its inputs are in, while later chunks'
 * inputs are still being copied, and its output is copied back as soon as the
 * kernel is done.  Page-locked host memory (cudaHostAlloc) lets the copies run
 * asynchronously at full speed; pageable memory works, more slowly.
 *
 *   dev_workspace  device memory of at least attn_fwd_host_workspace_size(dims)
 *                  bytes, 256-byte aligned, owned by the caller; it holds the
 *                  device copies of the tensors for the duration of the call.
 *   stream         caller's stream: the work is ordered after everything
 *                  already enqueued on it, and everything enqueued on it later
 *                  waits for the call's last copy back.  Internally the call
 *                  uses streams and events of its own (made once per device on
 *                  first use and kept for the life of the process).
 *
 * Asynchronous: returns once the work is enqueued; `out` holds the result once
 * `stream` is synchronised.  The host buffers and the workspace must stay valid
 * (and the inputs unchanged) until then.  Calls on different caller streams
 * must use different workspaces.
 *
 * Errors: as attn_fwd for dims, mask_kind and scale; NULL tensor or workspace
 * pointer (ATTN_ERR_NULL); workspace too small (ATTN_ERR_SHAPE) or not 256-byte
 * aligned (ATTN_ERR_ALIGN); out overlapping an input (ATTN_ERR_ALIAS); a
 * failing CUDA call (ATTN_ERR_CUDA; work enqueued before the failure may still
 * run, and the caller's stream still waits for it).  Host pointers need no
 * particular alignment.
 */
attn_status attn_fwd_host(const void *Q, const void *K, const void *V,
                          const int32_t *key_lengths, int mask_kind, float scale,
                          void *out, const attn_dims *dims, void *dev_workspace,
                          size_t dev_workspace_bytes, void *stream);

/*
 * attn_fwd that also writes each query row's log-sum-exp,
 *
 *     lse[b,h,i] = log sum_j exp( scale * Q[b,h,i,:] . K[b,h,j,:] + M[b,i,j] )
 *
 * (natural log; -inf for a row with no allowed key), so that the softmax
 * weights of the row are exp(s_ij - lse_i).  It is the statistic a backward
 * pass (attn_bwd) needs to recompute the weights without storing them.
 *
 *   lse   device float [B][h][m], 4-byte aligned, owned by the caller; must not
 *         overlap any other argument.
 * Other arguments, rules, errors and kernel choice as attn_fwd; lse NULL is
 * ATTN_ERR_NULL, unaligned ATTN_ERR_ALIGN, overlapping ATTN_ERR_ALIAS.
 */
attn_status attn_fwd_lse(const void *Q, const void *K, const void *V,
                         const int32_t *key_lengths, int mask_kind, float scale,
                         void *out, float *lse, const attn_dims *dims, void *stream);

/*
 * Restricted self-attention: attn_fwd where mask_kind may also hold
 * ATTN_MASK_WINDOW, which keeps, for query i, only the keys j with
 * |i - j| <= window (a neighbourhood of r = 2 * window + 1 positions around the
 * query; the deep-reading page's §04 complexity table lists "restricted
 * self-attention" at O(r n d), the slide deck's "Limitations and Future Work"
 * local, restricted attention).  The window combines with the other bits as a
 * union of masked keys (with CAUSAL: keys i - window .. i).  Key tiles outside
 * every row's window are never loaded or computed, so the work grows with
 * n * window, not n * n.
 *
 * Requires m == n when ATTN_MASK_WINDOW is set (ATTN_ERR_SHAPE) and window >= 0
 * (ATTN_ERR_VALUE).  Other arguments, rules, errors and kernel choice as attn_fwd;
 * without ATTN_MASK_WINDOW the call is attn_fwd.
 */
attn_status attn_fwd_window(const void *Q, const void *K, const void *V,
                            const int32_t *key_lengths, int mask_kind, int window, float scale,
                            void *out, const attn_dims *dims, void *stream);

/* Bytes of device workspace attn_bwd needs for these dims (host only, no CUDA
 * call); 0 if attn_bwd would reject the dims. */
size_t attn_bwd_workspace_size(const attn_dims *dims);

/*
 * Backward of the attention: with out = attn_fwd(Q, K, V) and an upstream
 * gradient dout of the same shape, the gradients of sum(dout * out),
 *
 *     dV = P^T dout,   dS = P o (dout V^T - D),   D_i = sum_c dout_ic out_ic,
 *     dQ = scale dS K, dK = scale dS^T Q,
 *
 * per (batch, head), P the softmax weights of the forward.  The pages train the
 * model (slide deck "Training Details") but do not write this pass out: it is
 * the chain rule of the attention equation.  P is recomputed from Q, K and lse.
 *
 *   Q, K, V, out   the forward's inputs and output (out as written by attn_fwd_lse)
 *   dout           device [B][h][m][d_k], the gradient of the loss w.r.t. out
 *   lse            device float [B][h][m] written by attn_fwd_lse for the same
 *                  inputs, mask and scale
 *   key_lengths, mask_kind, scale   as for the forward
 *   dQ, dK, dV     device outputs shaped like Q, K, V; every element is written
 *                  (0 for keys no query may see)
 *   workspace      device scratch of at least attn_bwd_workspace_size(dims)
 *                  bytes, 256-byte aligned, any contents; calls that may run at
 *                  the same time on the GPU need different workspaces
 *   dims, stream   as for the forward
 *
 * Supported: every dtype and head width attn_fwd takes.  bf16 with d_k a multiple of
 * 8 up to 64 runs on tensor cores (narrower heads zero-padded to 64 inside the
 * kernels; three kernels: a row pass for D and the padded per-row table that zeroes
 * the dQ accumulator, the tensor-core pass, the dQ conversion); fp32 and the other
 * bf16 widths up to 128 run on the CUDA cores with fp32 arithmetic (two kernels: a
 * rows pass for D and dQ, a keys pass for dK and dV).  All tensors
 * 16-byte aligned, lse 4-byte aligned (ATTN_ERR_ALIGN).  dQ, dK, dV and the
 * workspace must not overlap each other or any input (ATTN_ERR_ALIAS).  A
 * workspace that is too small is ATTN_ERR_SHAPE.  Other errors as attn_fwd.
 */
attn_status attn_bwd(const void *Q, const void *K, const void *V, const void *out,
                     const void *dout, const float *lse, const int32_t *key_lengths,
                     int mask_kind, float scale, void *dQ, void *dK, void *dV,
                     void *workspace, size_t workspace_bytes,
                     const attn_dims *dims, void *stream);

/* Bytes of device workspace attn_decode needs for these dims on the current
 * device (its SM count sets how the keys are split); 0 when no workspace is
 * needed or when attn_decode would reject the dims. */
size_t attn_decode_workspace_size(const attn_dims *dims);

/*
 * Incremental decoding: m (1..8) new query rows per (batch, head) against a
 * cache of keys and values, as when a decoder produces one position at a time
 * and attends to the positions produced so far ("Paper Deep Reading", §03
 * "Decoder layer").  Query i of batch b sees cached keys 0 .. cache_lengths[b]-1:
 * exactly attn_fwd with ATTN_MASK_KEY_PADDING and key_lengths = cache_lengths
 * (a row with no cached key is 0).
 *
 *   Q              device bf16 [B][h][m][d_k], 1 <= m <= 8, d_k in {16, 32, 64, 128} (the
 *                  head widths of the model-variant table)
 *   K, V           device bf16 [B][h][n][d_k]: the caches, n = their capacity
 *   cache_lengths  device int32 [B], clamped to [0, n]; NULL: every row holds n keys
 *   scale          as for attn_fwd
 *   out            device bf16 [B][h][m][d_k]
 *   lse            NULL, or device float [B][h][m]: each row's log-sum-exp (natural log)
 *   workspace      attn_decode_workspace_size(dims) bytes, 16-byte aligned, any
 *                  contents (may be NULL when that size is 0); calls that may run
 *                  at the same time on the GPU need different workspaces
 *
 * The keys of each (batch, head) are split over several CTAs on the CUDA cores
 * (the work is memory-bound: each cached row is read once per call), then one
 * pass merges the splits.  Errors as attn_fwd, plus: dtype other than bf16 or
 * another d_k (ATTN_ERR_DTYPE), m > 8 (ATTN_ERR_SHAPE), workspace NULL or too small
 * when one is needed (ATTN_ERR_NULL / ATTN_ERR_SHAPE), lse or the workspace
 * unaligned (ATTN_ERR_ALIGN) or overlapping a tensor (ATTN_ERR_ALIAS).
 */
attn_status attn_decode(const void *Q, const void *K, const void *V, const int32_t *cache_lengths,
                        float scale, void *out, float *lse, const attn_dims *dims,
                        void *workspace, size_t workspace_bytes, void *stream);

/* Shapes of a multi-head attention call with its projections (d_v = d_k). */
typedef struct {
    int32_t B;       /* batch */
    int32_t h;       /* heads; h * d_k must be a multiple of 128 */
    int32_t m;       /* query positions */
    int32_t n;       /* key/value positions */
    int32_t d_model; /* model width, a multiple of 128 */
    int32_t d_k;     /* head width: a multiple of 8 up to 64, or 128 (0 is read as 64); the
                        pages' d_model / h */
} attn_mha_dims;

/* Bytes of device workspace attn_mha_fwd needs (host only, no CUDA call); 0 if
 * attn_mha_fwd would reject the dims. */
size_t attn_mha_workspace_size(const attn_mha_dims *dims);

/*
 * Multi-head attention with its projections ("Paper Deep Reading", §04; the
 * slide deck's "Multi-Head Attention" slide; heads of width 64, as in the base and
 * big models, or 128, the model-variant table's h = 4 row):
 *
 *     head_i = Attention(Xq W_i^Q, Xkv W_i^K, Xkv W_i^V),
 *     out    = Concat(head_1, ..., head_h) W^O,
 *
 * with d_k = d_v = dims->d_k and no bias terms (the formula has none); Attention
 * is attn_fwd's (mask and scale as there; ATTN_SCALE_DEFAULT gives 1/sqrt(d_k)).
 * All tensors bf16, row-major, in device memory of the current device, 16-byte
 * aligned:
 *   Xq   [B][m][d_model], Xkv [B][n][d_model] (pass Xq for self-attention)
 *   Wq, Wk, Wv  [d_model][h * d_k]: head i uses columns i d_k .. (i + 1) d_k - 1
 *   Wo   [h * d_k][d_model]: head i's output multiplies rows i d_k .. (i + 1) d_k - 1
 *   out  [B][m][d_model]
 *   workspace  attn_mha_workspace_size(dims) bytes (Q, K, V and the heads'
 *              outputs in [B][h][len][d_k], and for narrow heads the concatenated
 *              projections), 256-byte aligned, any contents
 * With d_k 64 or 128, three kernels are enqueued: the three projections into the
 * head-split layout (one tcgen05 GEMM launch whose epilogue writes each 64-column
 * block into its head), the attention, and the output projection, which reads the
 * heads' outputs as its K dimension directly (the concatenation costs no copy).
 * Narrower heads (the model-variant table's 16 and 32) take the projections into
 * the concatenated layout [B][len][h * d_k], copy them into heads and the heads'
 * outputs back (memory-bound copies), with the attention in between.
 *
 * Errors: NULL pointers (ATTN_ERR_NULL), bad shapes or h * d_k or d_model not
 * multiples of 128, causal with m != n (ATTN_ERR_SHAPE), d_k not a multiple of 8 up
 * to 64 and not 128 (ATTN_ERR_DTYPE), mask bits other than
 * KEY_PADDING and CAUSAL (ATTN_ERR_MASK), unaligned pointers (ATTN_ERR_ALIGN),
 * bad scale (ATTN_ERR_VALUE), a workspace too small (ATTN_ERR_SHAPE), out or the
 * workspace overlapping an input or each other (ATTN_ERR_ALIAS), CUDA errors.
 */
attn_status attn_mha_fwd(const void *Xq, const void *Xkv, const void *Wq, const void *Wk,
                         const void *Wv, const void *Wo, const int32_t *key_lengths,
                         int mask_kind, float scale, void *out, const attn_mha_dims *dims,
                         void *workspace, size_t workspace_bytes, void *stream);

/* The kernel attn_fwd would run for these dims and mask (host only, no CUDA call);
 * ATTN_KERNEL_AUTO (0) if the call would be rejected. */
int attn_select_kernel(const attn_dims *dims, int mask_kind);

/*
 * Synchronises `stream`, then reports whether any kernel of this library on
 * the current device gave up a bounded wait since the previous call
 * (ATTN_ERR_DEVICE_TIMEOUT; *info, if not NULL, receives a code naming the
 * wait) or not (ATTN_OK).  Clears the record.  ATTN_ERR_CUDA if the
 * synchronisation itself fails.  A kernel that gives up a wait stops early and
 * leaves its output incomplete, but leaves the CUDA context usable.
 */
attn_status attn_device_status(void *stream, int32_t *info);

/*
 * Test hook of the failure detection (not part of the operation; no page of the
 * method has a counterpart).  Runs the whole-head-resident kernel of attn_fwd on
 * these arguments with every bounded wait limited to wait_ns nanoseconds and with
 * the barrier on which the rows report their first chunk of weights stored waiting
 * for one report more than they make (one arrival withheld), so the MMA-issuing
 * thread's wait for that chunk runs out: the kernel records the
 * time-out (attn_device_status then returns ATTN_ERR_DEVICE_TIMEOUT with info 403,
 * the weights wait of that kernel), waits for its own copies and MMAs, frees its
 * TMEM and exits without writing `out`.  The CUDA context stays usable.  It lets a
 * test check the abort path without any fault on the GPU.
 *
 * Arguments as attn_fwd; the dims must be ones the resident kernel runs (bf16, d_k a
 * multiple of 8 up to 64, n <= 256; ATTN_ERR_UNSUPPORTED otherwise);
 * wait_ns in [100000, 2000000000] (ATTN_ERR_VALUE otherwise).
 */
attn_status attn_test_withheld_arrival(const void *Q, const void *K, const void *V,
                                       const int32_t *key_lengths, int mask_kind, float scale,
                                       void *out, const attn_dims *dims, uint64_t wait_ns,
                                       void *stream);

/* Static description of a status code (never NULL). */
const char *attn_status_string(int status);

/* ABI version: (major << 16) | minor. */
int32_t attn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_GB300_ATTN_H */
