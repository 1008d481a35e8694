/*
 * attnres.h -- C ABI of the Blocked Attention Residuals layer in libkda.
 *
 * The operation ("Kimi (AI)", Wikipedia mirror, section "Attention
 * Residuals"): layer i of a network takes as input a softmax attention over
 * depth, h_i = SoftmaxAttention(q_i, K_i, V_i), with one learned query q_i
 * per layer and K_i = V_i the list of earlier outputs.  In the blocked form
 * the layers are cut into consecutive blocks and layer i of block n attends
 * over the sums of the outputs of every earlier block and, from the block's
 * second layer on, the sum of its own block's earlier outputs.  The network
 * input counts as block 0 (a block of one output), so that the first layer
 * has a source.  Attention runs per token, independently: for token t,
 *
 *     h[t] = sum_j w_j[t] s_j[t],   w[t] = softmax_j(scale * q . s_j[t]).
 *
 * Conventions as in kda.h: device pointers owned by the caller, 16-byte
 * aligned, row-major, work enqueued on `stream`, argument errors returned
 * synchronously before any launch.
 */
#ifndef ATTNRES_H_
#define ATTNRES_H_

#include "kda.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * One layer's input under Blocked Attention Residuals, for T tokens of width d.
 *
 *   blocks      [num_blocks][T][d] (dtype): sums of the finished blocks'
 *               outputs, block 0 (the network input) first
 *   partial     [T][d] fp32 or NULL: sum of the current block's outputs
 *               before the previous layer
 *   h_last      [T][d] (dtype) or NULL: the previous layer's output
 *   partial_out [T][d] fp32 or NULL: receives P = partial + h_last; may equal
 *               partial (the running sum updated in place)
 *   block_out   [T][d] (dtype) or NULL: receives P rounded to dtype (at a
 *               block's first layer P is the finished block's sum, to be
 *               stored as the next entry of `blocks`)
 *   q           [d] fp32: the layer's query
 *   scale       logit scale; 1/sqrt(d) gives standard scaled dot-product
 *               attention
 *   h           [T][d] (dtype) output: the layer's input
 *
 * The sources are blocks[0 .. num_blocks-1], then P when partial or h_last
 * is given (P in fp32).  Softmax and sums are fp32.  partial_out and
 * block_out need partial or h_last.  No output may overlap an input or
 * another output, except partial_out == partial.
 *
 * Supported: dtype KDA_BF16 or KDA_FP32, d a multiple of 8, 1 to 64 sources.
 * T == 0 is a valid no-op.
 *
 * Returns, before any launch: KDA_ERR_INVALID_ARG for a negative count or
 * size, an unknown dtype, no source at all, partial_out or block_out without
 * partial or h_last, a missing q, h or (num_blocks > 0) blocks, a pointer not
 * 16-byte aligned, or overlapping buffers; KDA_ERR_UNSUPPORTED for d not a
 * multiple of 8 or more than 64 sources.  KDA_ERR_CUDA if the launch fails.
 * The kernel has no data-dependent error: any finite inputs give a result.
 */
kda_status attnres_layer(const void* blocks, int32_t num_blocks, const float* partial,
                         const void* h_last, float* partial_out, void* block_out,
                         const float* q, float scale, int64_t T, int32_t d, kda_dtype dtype,
                         void* h, kda_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* ATTNRES_H_ */
