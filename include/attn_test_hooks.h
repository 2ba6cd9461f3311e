/*
 * attn_test_hooks.h -- the extra entry point of the test-hook build, libattn_testhooks.so (the
 * kernels of libattn.so compiled with -DATTN_TEST_HOOKS; libattn.so neither exports this nor
 * carries its kernel parameter). Every entry point of attn.h is exported by this build too and
 * behaves the same. Nothing a user needs calls it: it exists so that the tests can make the
 * kernel's bounded waits run out without any GPU fault.
 */
#ifndef GB300_ATTN_TEST_HOOKS_H
#define GB300_ATTN_TEST_HOOKS_H

#ifdef __cplusplus
extern "C" {
#endif

/*
 * attn_fwd_withhold -- runs attn_fwd (dense, its default rebase threshold) except that every CTA's TMA
 * producer skips K/V token `token` (token 2i is K tile i, token 2i+1 is V tile i, tiles of 128
 * keys), so the waits that need it never complete. About two seconds after launch the first
 * such wait gives up and records its status word (see attn_device_status); every CTA then
 * drains its own loads and MMAs, frees its tensor memory and exits, and the context stays
 * usable. O and lse are left undefined.
 *
 *   token : 0 <= token < 2 * ceil(S / 128), else ATTN_ERR_INVALID_ARG.
 * Other arguments, errors and ownership as attn_fwd.
 */
int attn_fwd_withhold(const void* q, const void* k, const void* v, void* o, float* lse,
                      int B, int H, int S, int D, float scale, int token, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* GB300_ATTN_TEST_HOOKS_H */
