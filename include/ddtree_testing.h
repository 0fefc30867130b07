/*
 * ddtree_testing.h - test-only entry points of libddtree.so.
 *
 * Not part of the verify-step ABI (include/ddtree.h); a serving caller never
 * needs these. They exist so that tests can drive failure paths of the
 * kernels without faulting or hanging the GPU.
 */
#ifndef DDTREE_TESTING_H
#define DDTREE_TESTING_H

#include <stddef.h>
#include <stdint.h>

#include "ddtree.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * ddtree_testing_attn_stall - tree_verify_attn with one bounded wait made to
 * run out.
 *
 * Arguments are tree_verify_attn's, plus stall_ns (1 .. 1e9). In every CTA of
 * the tensor-core attention kernel, the warp that issues row tile 0's MMAs
 * first waits on an mbarrier that nothing completes, with a limit of
 * stall_ns nanoseconds instead of the normal two seconds. The wait gives up,
 * sets the CTA's abort flag and DDT_DEV_TIMEOUT in *dev_status; every other
 * wait in the CTA then stops at once, the copies and MMAs already issued are
 * drained (under their normal limits, so none is left in flight), TMEM is
 * freed and the CTA returns. Rows whose work was cut short get zeros (lse
 * -inf); rows that finished before the abort keep their results. The
 * call returns DDT_OK after the launches, like tree_verify_attn; the timeout
 * is seen in *dev_status after the stream is synchronised, and the next call
 * on the same context runs normally.
 *
 * Only the tensor-core kernel (Dh 128, Hq/Hkv dividing 128, R <= 264 rows,
 * scale > 0) has bounded waits; other shapes return DDT_ESHAPE.
 * DDT_EINVAL for stall_ns == 0 or above one second.
 */
int ddtree_testing_attn_stall(const ddtree_bf16* q, const ddtree_bf16* k_tree,
                              const ddtree_bf16* v_tree, const ddtree_bf16* k_cache,
                              const ddtree_bf16* v_cache, int num_pages, int page_size,
                              const int32_t* page_table, int max_pages, const int32_t* ctx_len,
                              const uint32_t* vis, const int32_t* n_nodes, int B, int N, int Hq,
                              int Hkv, int Dh, float scale, ddtree_bf16* out, float* lse,
                              void* workspace, size_t workspace_bytes, int32_t* dev_status,
                              void* stream, uint64_t stall_ns);

/*
 * ddtree_testing_gumbel - the Gumbel noise the temperature walks add to each
 * token's scaled logit for the bonus draw ("The Architecture of Speculative
 * Decoding", Section 3: the bonus comes from the residual distribution, drawn
 * here as a Gumbel-max), for given Philox words.
 *
 * words (device, n uint32): Philox output words; U = ((w >> 8) + 0.5) 2^-24.
 * out (device, n fp32): g = -log(-log U) as the walks compute it in fp32.
 * Returns DDT_OK (n == 0: nothing runs), DDT_EINVAL for NULL pointers,
 * DDT_ECUDA if the launch fails. Asynchronous on `stream`.
 */
int ddtree_testing_gumbel(const uint32_t* words, float* out, size_t n, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* DDTREE_TESTING_H */
