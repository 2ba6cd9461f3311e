/*
 * attn.h -- C ABI of the GB300 (sm_103a) dense attention forward library (libattn.so).
 *
 * The operation (the pages: "B200 attention kernel from scratch to ~SOTA in 60 figures
 * (CUDA/PTX)", Ch. 1 §ii "work parallelisation" and §B "online softmax"): for every batch b,
 * head h and query row i < S, over all keys j < S (dense, non-causal, no mask),
 *
 *     s_ij   = scale * sum_d Q[b,h,i,d] * K[b,h,j,d]
 *     O[b,h,i,:] = sum_j softmax_j(s_i.) * V[b,h,j,:]
 *     lse[b,h,i] = ln sum_j exp(s_ij)          (natural log, fp32)
 *
 * The pages fix the scope: BF16 inputs, head_dim 128, dense, non-causal. lse is not on the
 * pages; it is the usual FlashAttention by-product (natural log of the row's softmax
 * denominator over the scaled scores).
 *
 * Thread safety: every entry point may be called from several host threads at once.
 */
#ifndef GB300_ATTN_H
#define GB300_ATTN_H

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes returned by every entry point. */
typedef enum {
    ATTN_OK = 0,
    ATTN_ERR_INVALID_ARG = 1,        /* null pointer, non-positive size, bad scale, overlap, overflow */
    ATTN_ERR_UNSUPPORTED_DIM = 2,    /* D != 128 */
    ATTN_ERR_MISALIGNED = 3,         /* q/k/v/o not 16-byte aligned, or lse not 4-byte aligned */
    ATTN_ERR_UNSUPPORTED_DEVICE = 4, /* no CUDA device, or the current device is not sm_103 */
    ATTN_ERR_LAUNCH = 5,             /* tensor-map encoding or kernel launch failed */
    ATTN_ERR_TIMEOUT = 6             /* a kernel gave up a bounded wait: attn_device_status returns the
                                        word; the Python binding's check_device_status raises this code */
} attn_status;

/*
 * attn_fwd -- O = softmax(scale * Q K^T) V and lse, one fused kernel launch.
 *
 *   q, k, v : DEVICE pointers, BF16, contiguous [B, H, S, D] (row = one (b,h,s), 256 bytes).
 *             Read only. 16-byte aligned.
 *   o       : DEVICE pointer, BF16, contiguous [B, H, S, D], written. 16-byte aligned. Must not
 *             overlap q, k, v or lse.
 *   lse     : DEVICE pointer, fp32 [B, H, S], written (natural log); 4-byte aligned. May be
 *             NULL, in which case lse is not written.
 *   B, H, S : batch, heads, sequence length; each >= 1, and B*H*ceil(S/256) <= 2^31 - 1.
 *             S need not be a multiple of 128: padded keys contribute nothing and padded
 *             query rows are never written.
 *   D       : head dimension; must be 128.
 *   scale   : softmax scale applied to Q K^T (usually 1/sqrt(D)); finite and > 0. (The kernel
 *             takes the row max on raw scores and multiplies it by the scale afterwards, as
 *             the pages' Ch. 8 does, which is only valid for a positive scale.)
 *   stream  : a cudaStream_t (NULL = the legacy default stream). The call is asynchronous:
 *             it enqueues one kernel and returns; nothing is synchronised on the host.
 *
 * Resources: the kernel launches min(B*H*ceil(S/256), number of SMs) CTAs of 512 threads, each
 * holding one SM's tensor memory and ~227 KB of its shared memory, and each working through
 * its share of the work items (256 query rows of one (b, h) against all of that head's keys).
 *
 * Ownership: all buffers belong to the caller. The library allocates no device memory and
 * keeps no per-call state; it caches only per-device launch attributes.
 *
 * Errors: arguments are checked before any CUDA call; on any error nothing is launched and
 * o / lse are untouched. A launch failure is reported as ATTN_ERR_LAUNCH (the CUDA error is
 * not cleared for the caller). Faults that happen while the kernel runs surface, as usual,
 * at the caller's next synchronisation; a kernel that gave up a bounded internal wait
 * records it in the device status word read by attn_device_status().
 */
int attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
             int B, int H, int S, int D, float scale, void* stream);

/*
 * attn_fwd_ex -- attn_fwd with the online-softmax rebase threshold chosen by the caller
 * ("B200 attention kernel from scratch to ~SOTA in 60 figures (CUDA/PTX)", Ch. 11
 * "skip O rescale"): the kept row max, and with it the scaling of O and of the row sum, moves
 * only when a K/V tile's max exceeds it by at least the threshold, in base-2 exponent units.
 * The result does not depend on it beyond rounding.
 *
 *   rebase_threshold_log2 = 1 : what attn_fwd, attn_fwd_causal and attn_fwd_host use; P <= 2,
 *                               one fp32 row sum normalises O and gives lse.
 *   rebase_threshold_log2 = 0 : the kept row max is the running max; P <= 1.
 *   rebase_threshold_log2 = 8 : the pages' choice; P may reach 2^8 and the output is
 *                               normalised by the sum of the BF16-rounded P.
 * Any other value: ATTN_ERR_INVALID_ARG. All other arguments, errors and ownership as attn_fwd.
 */
int attn_fwd_ex(const void* q, const void* k, const void* v, void* o, float* lse,
                int B, int H, int S, int D, float scale, int rebase_threshold_log2,
                void* stream);

/*
 * attn_fwd_causal -- attn_fwd with the causal mask: query i attends to keys j <= i only
 * (queries and keys share the positions 0..S-1), so every max, sum and product in the
 * definition above runs over j <= i. Not on the pages, whose scope is non-causal; this is the
 * usual decoder mask. The kernel visits only the K/V tiles at or before each Q tile's
 * diagonal (about half the work of attn_fwd at large S). Arguments, errors and ownership as
 * attn_fwd.
 */
int attn_fwd_causal(const void* q, const void* k, const void* v, void* o, float* lse,
                    int B, int H, int S, int D, float scale, void* stream);

/*
 * attn_fwd_strided -- attn_fwd_ex on strided tensors (no copies): [B, S, H, D], slices of a
 * packed QKV buffer, and so on. The head dimension must be contiguous (unit stride).
 *
 *   q_strides, k_strides, v_strides, o_strides : HOST pointers to 3 element strides each,
 *             {batch, head, sequence}; element (b, h, s, d) of q is q + b*qs[0] + h*qs[1] +
 *             s*qs[2] + d. Every stride must be > 0 and a multiple of 8 elements (16 bytes,
 *             a TMA requirement); the output strides must not map two elements to one
 *             address. Read during the call only.
 *   lse     : still a contiguous fp32 [B, H, S] (or NULL).
 *   Overlap between o / lse and the inputs is checked on the address ranges the strides span.
 *   Contiguous [B, H, S, D] corresponds to strides {H*S*D, S*D, D}; [B, S, H, D] to
 *   {S*H*D, D, H*D}.
 *   causal  : 0 = dense (attn_fwd_ex), 1 = causal mask (attn_fwd_causal); anything else is
 *             ATTN_ERR_INVALID_ARG.
 * Other arguments, errors and ownership as attn_fwd_ex.
 */
int attn_fwd_strided(const void* q, const void* k, const void* v, void* o, float* lse,
                     int B, int H, int S, int D, float scale,
                     const long long* q_strides, const long long* k_strides,
                     const long long* v_strides, const long long* o_strides,
                     int rebase_threshold_log2, int causal, void* stream);

/*
 * attn_fwd_host -- attn_fwd (or attn_fwd_causal) from HOST buffers to HOST buffers: enqueues on
 * `stream` the copies of q_h, k_h, v_h into the caller's device buffers q_d, k_d, v_d, the
 * kernel, and the copies of o_d and lse_d back into o_h and lse_h, then returns. Synchronise
 * the stream before reading o_h / lse_h or reusing any of the buffers.
 *
 *   q_h, k_h, v_h : HOST pointers, BF16, contiguous [B, H, S, D]; read by the copies.
 *   o_h           : HOST pointer, BF16 [B, H, S, D], written by the copy-out.
 *   lse_h         : HOST pointer, fp32 [B, H, S], or NULL (then lse_d must be NULL too).
 *   q_d .. lse_d  : DEVICE buffers of the same shapes, owned by the caller, with attn_fwd's
 *                   alignment rules; the library allocates nothing. No two of the five may
 *                   overlap: unlike attn_fwd's inputs, q_d, k_d and v_d are written (by the
 *                   copy-in), so they may not alias one another either.
 *   causal        : 0 = attn_fwd, 1 = attn_fwd_causal.
 * Host buffers should be page-locked (cudaHostAlloc, or a pinned torch tensor) for the copies
 * to run asynchronously and overlap other streams; pageable memory still works, with the
 * CUDA runtime's staging.
 * Errors: every check attn_fwd makes is made before anything is enqueued, plus NULL host
 * pointers, an lse_h / lse_d mismatch and overlapping q_d / k_d / v_d (ATTN_ERR_INVALID_ARG);
 * a failed copy is ATTN_ERR_LAUNCH.
 */
int attn_fwd_host(const void* q_h, const void* k_h, const void* v_h, void* o_h, float* lse_h,
                  void* q_d, void* k_d, void* v_d, void* o_d, float* lse_d,
                  int B, int H, int S, int D, float scale, int causal, void* stream);

/*
 * attn_fwd_host_noalloc -- attn_fwd_host for callers that cannot allocate device memory (code
 * that may not call cudaMalloc because another allocator owns the device memory of the process,
 * or that runs where allocations are forbidden). The pages have no counterpart: this is a
 * convenience of this library's boundary, not a step of the method.
 *
 * The device staging that attn_fwd_host takes from its caller (q_d .. lse_d) is instead a fixed
 * array inside the library, ATTN_NOALLOC_MAX_ROWS rows of q, k, v, o and lse (33,685,504 bytes),
 * held on every GPU where the library's device code is loaded until the process exits. The call
 * allocates nothing: no cudaMalloc, no cudaFree, no allocating library routine.
 *
 *   q_h .. lse_h, B, H, S, D, scale, causal, stream : as attn_fwd_host (lse_h may be NULL).
 *   B * H * S must not exceed ATTN_NOALLOC_MAX_ROWS (e.g. B = 1, H = 8, S = 4096), else
 *   ATTN_ERR_INVALID_ARG before anything is enqueued.
 *
 * Set-up: the first call on a device (with that device current) looks up the array's device
 * address with cudaGetSymbolAddress, which may load the library's device code; make that first
 * call before any stream capture. Later calls only enqueue the copies and the kernel.
 * Sharing: every call uses the same array, which keeps the last call's contents; nothing in it
 * needs clearing, since each call overwrites whatever it reads. Calls whose work overlaps on
 * the GPU (different streams, not ordered by events or synchronisation) race on the array and
 * corrupt each other's results: order them, e.g. one stream.
 * Errors: as attn_fwd_host; ATTN_ERR_UNSUPPORTED_DEVICE also when the current device is not
 * sm_103, ATTN_ERR_LAUNCH when the array's address cannot be obtained.
 */
#define ATTN_NOALLOC_MAX_ROWS 32768
int attn_fwd_host_noalloc(const void* q_h, const void* k_h, const void* v_h, void* o_h, float* lse_h,
                          int B, int H, int S, int D, float scale, int causal, void* stream);

/* A short, static, human-readable description of a status code. Never NULL. */
const char* attn_status_string(int status);

/*
 * attn_device_status -- read (and optionally clear) the current device's status word.
 *
 * The attention kernel bounds every internal wait (about two seconds). A CTA that gives up
 * stops its work, releases its tensor memory, leaves its outputs incomplete and records a
 * non-zero word here (the first failure wins). Call it after synchronising the streams that
 * ran attn_fwd. *word receives 0 when no wait gave up. Returns ATTN_OK, or
 * ATTN_ERR_UNSUPPORTED_DEVICE / ATTN_ERR_LAUNCH if the word could not be read.
 *
 * Word layout: 0xA77E0000 | role << 8 | barrier, role 1 = TMA producer, 2 = MMA issue,
 * 3 = softmax, 4 = O correction; barrier = the index of the mbarrier whose wait ran out
 * (0-17), or 18 + q for the producer's wait on the count of Q tile q's S tiles that the
 * softmax warps have taken.
 */
int attn_device_status(unsigned int* word, int reset);

/* Library version, (major << 16) | minor. */
int attn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* GB300_ATTN_H */
