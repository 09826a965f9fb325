/*
 * mla_absorb.h — C ABI of the weight-absorption batched GEMMs that sit on
 * either side of absorbed-MLA decode attention (libmla_decode.so).
 *
 * The operations ("DeepSeek V3/R1 Inference Efficiency (2): Reverse-
 * Engineering the Production Deployment", §2.4.1, Compute)
 * ------------------------------------------------------------------------
 * QKV projection, Q''' = bmm(Q'', W_UK^T), bmm([n_head, bs, 128],
 * [n_head, 128, 512]): with the key up-projection absorbed into the query,
 * each head's 128 "nope" query dims are mapped into the 512-dim latent space
 * the cache rows live in, so that attention can score latent rows directly:
 *
 *     q_latent[t, h, c] = sum_d q_nope[t, h, d] * W_UK[h, c, d]
 *
 * O projection, O' = bmm(PV, W_UV), [n_head, bs, c] @ [n_head, c, d]: the
 * value up-projection is applied once to the attention output:
 *
 *     out[t, h, d] = sum_c O[t, h, c] * W_UV[h, c, d]
 *
 * with c = 512 latent dims, d = 128 per-head dims, t over the T tokens of
 * the step (request x query token), h over the heads.  Both weights are in
 * the pages' [n_head, c = 512, d = 128] layout, d contiguous (a checkpoint
 * that stores the up-projection per head as [d, c] is transposed once when
 * it is loaded).  Inputs and outputs are bf16; products accumulate in fp32
 * on the tensor cores and are rounded to bf16 once.
 *
 * Layout
 * ------
 * A token-major activation holds row (t, h) at element (t * num_heads + h) *
 * stride; the row's dims are contiguous.  That is the layout the decode
 * attention reads its query from (stride 576: latent dims 0..511, RoPE dims
 * 512..575) and writes its output to (stride 512), so the query-side call
 * can write the attention's query in place and the output-side call can read
 * the attention's output directly.
 *
 * Conventions (as for the decode calls)
 * -------------------------------------
 *  - Every pointer is a DEVICE pointer, 16-byte aligned; strides are in
 *    elements, multiples of 8 (16 bytes).  Outputs must not overlap inputs.
 *  - The return value reports errors found on the host (MLA_ERR_INVALID_ARG
 *    for bad pointers, sizes or strides; MLA_ERR_UNSUPPORTED for a head count
 *    outside 1..128; MLA_ERR_DEVICE off a compute capability 10.3 device;
 *    MLA_ERR_CUDA for a launch failure).  num_tokens == 0 launches nothing.
 *  - `status` is a device int that the kernels set to MLA_ERR_TIMEOUT (from
 *    0, atomically) if one of their bounded waits runs out, leaving their
 *    outputs unspecified; the calls never clear it.  mla_workspace_status()
 *    reads it (it reads word 0 of the buffer it is given).
 *  - Asynchronous on `stream`, no allocation, no host synchronisation;
 *    graph-capturable.  Thread-safe.
 */
#ifndef MLA_ABSORB_H_
#define MLA_ABSORB_H_

#include "mla_decode.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Query-side absorption.
 *   q_nope     bf16, row (t, h) at q_nope + (t * num_heads + h) * q_stride,
 *              128 dims.
 *   q_pe       bf16 or NULL, row (t, h) at q_pe + (t * num_heads + h) *
 *              q_stride, 64 RoPE dims; copied unchanged to dims 512..575 of
 *              the output row.  (With the usual [T, H, 192] projection
 *              output, q_nope = base, q_pe = base + 128, q_stride = 192.)
 *   q_stride   >= 128 (>= 64 for q_pe), multiple of 8.
 *   w_uk       bf16 [num_heads, 512, 128] (W_UK[h, c, d]), contiguous.
 *   out        bf16, row (t, h) at out + (t * num_heads + h) * out_stride:
 *              dims 0..511 = q_latent, 512..575 = q_pe (when given).
 *   out_stride >= 512, or >= 576 with q_pe; multiple of 8.  576 writes the
 *              decode attention's query [T, num_heads, 576] directly.  */
int mla_absorb_q(const void* q_nope, const void* q_pe, int64_t q_stride, const void* w_uk,
                 int num_tokens, int num_heads, void* out, int64_t out_stride, int* status,
                 mla_stream_t stream);

/* Output-side absorption.
 *   o          bf16, row (t, h) at o + (t * num_heads + h) * o_stride, 512
 *              latent dims (the decode attention's bf16 output has
 *              o_stride = 512).
 *   o_stride   >= 512, multiple of 8.
 *   w_uv       bf16 [num_heads, 512, 128] (W_UV[h, c, d]), contiguous.
 *   out        bf16, row (t, h) at out + (t * num_heads + h) * out_stride,
 *              128 dims.
 *   out_stride >= 128, multiple of 8 (128 gives the [T, num_heads * 128]
 *              input of the output projection).  */
int mla_absorb_o(const void* o, int64_t o_stride, const void* w_uv, int num_tokens, int num_heads,
                 void* out, int64_t out_stride, int* status, mla_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MLA_ABSORB_H_ */
