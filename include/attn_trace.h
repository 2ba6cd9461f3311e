/*
 * attn_trace.h -- extra entry points of the trace build, libattn_trace.so (the same kernels as
 * libattn.so compiled with -DATTN_TRACE; libattn.so does not export these). Every other entry
 * point of attn.h is exported by the trace build too and behaves the same.
 *
 * The trace build records, for each CTA index below its capacity (4096 CTAs), sixteen 64-bit
 * words from the GPU's global nanosecond timer. A CTA walks several work items (pairs of Q
 * tiles); words 2-4 belong to its first item:
 *   0 CTA entry, 1 setup done (barriers initialised, tensor memory allocated),
 *   2 Q tile 0's first S seen by the softmax, 3 O tile 0 complete, 4 O tile 1 complete,
 *   5 before the final CTA barrier (after the CTA's last item), 6 the SM id (not a time),
 *   7 CTA exit;
 * words 8-15 are the boundary between the CTA's first two items, for Q tile 0:
 *   8 the first item's last S seen, 9 its last part of P stored, 10 its O read out of tensor
 *   memory (O released to the next item), 11 its epilogue done, 12 the next item's first S
 *   seen, 13 the next item's first part of P stored, 14 the next item's first QK issued,
 *   15 the next item's first PV issued (14 and 15 by the issuing warp).
 * A word is 0 if that point was not reached (or the CTA index is beyond the capacity; words
 * 12-15 when the CTA has one item). Each launch overwrites the words of the CTAs it runs.
 */
#ifndef GB300_ATTN_TRACE_H
#define GB300_ATTN_TRACE_H

#ifdef __cplusplus
extern "C" {
#endif

/* Copy the words of the first max_ctas CTAs (at most 4096) to the HOST buffer out
 * (16 * max_ctas entries). Call after synchronising the stream of the traced launch.
 * Returns ATTN_OK, ATTN_ERR_INVALID_ARG (null out, max_ctas <= 0) or ATTN_ERR_LAUNCH. */
int attn_trace_read(unsigned long long* out, int max_ctas);

/* Zero every word (synchronous). Returns ATTN_OK or ATTN_ERR_LAUNCH. */
int attn_trace_clear(void);

#ifdef __cplusplus
}
#endif

#endif
