/*
 * attnres.h - C ABI of the GB300 (sm_103a) AttnRes depth-wise aggregation.
 *
 * Attention Residuals replace the additive residual of a pre-norm Transformer
 * with a softmax-weighted sum over depth. For one token and one read (the
 * input of one sublayer, or of the LM head):
 *
 *     e_i = w^T RMSNorm_key(v_i)              (no 1/sqrt(d), temperature 1)
 *     a_i = exp(e_i) / sum_j exp(e_j)
 *     z   = sum_i a_i v_i
 *
 * (DepthBench reading notes, section 2.3 "Full AttnRes", paper Appendix A;
 * LLMRes blog, section "Kimi AttnRes": phi(q, k) = exp(q^T RMSNorm(k)),
 * q = w_l, k_i = v_i, with RMSNorm applied to the keys only.) RMSNorm is not
 * written out on the pages; this library uses the plain form
 * RMSNorm(x)_k = gamma_k x_k / sqrt(mean_k x_k^2 + eps).
 *
 * Full AttnRes: the sources of read l are the embedding v_0 and every earlier
 * sublayer output. Block AttnRes (DepthBench reading notes section 2.5; LLMRes
 * blog "Block Attention Residuals"; datacamp explainer "block attention
 * residuals"): the sublayers are cut into blocks of S; a read attends over the
 * embedding, the sums of the completed blocks, and the running sum of the
 * current block when it is non-empty. The two-stage computation (datacamp
 * explainer, "two-stage computation") batches the S pseudo-queries of a block
 * against the cross-block sources (stage 1) and folds in the running sum with
 * an online-softmax merge (stage 2).
 *
 * Conventions for every entry point:
 *   - Pointers named as device pointers must point to device memory of the
 *     current CUDA device; the library reads and writes them only from
 *     kernels. Host arrays are marked "host".
 *   - The caller owns all memory. The library keeps no per-call state and
 *     allocates no device memory.
 *   - Work is enqueued on `stream` (a cudaStream_t passed as void*; NULL is
 *     the legacy default stream) and is asynchronous: the call returns before
 *     the kernels finish. No call synchronises, except attnres_device_status.
 *   - Tensors are row-major. A [T, d] tensor has row stride d (contiguous);
 *     "sources" of a read are consecutive [T, d] slices `src_stride` elements
 *     apart, src_stride >= T*d.
 *   - dtype arguments take attnres_dtype values. Storage is fp32 or bf16;
 *     arithmetic is fp32 throughout; bf16 results are rounded to nearest even.
 *     w and gamma are always fp32; eps is a host scalar (>= 0).
 *   - T == 0 is valid and launches nothing.
 *   - Fast kernels need 16-byte aligned pointers and d a multiple of 128
 *     (full read), of the per-warp slice (stage 1) or of 8 (merge); any other
 *     valid input runs on a general kernel with the same results.
 *   - Errors: ATTNRES_ERR_INVALID_ARG for bad arguments (nothing launched),
 *     ATTNRES_ERR_UNSUPPORTED for valid requests beyond a stated limit,
 *     ATTNRES_ERR_CUDA when a launch fails (the CUDA error is consumed).
 *     Device-side waits are bounded; a wait that runs out makes the kernel
 *     stop and is reported by attnres_device_status as ATTNRES_ERR_TIMEOUT.
 *   - Outputs must not overlap inputs unless a function says otherwise.
 */
#ifndef ATTNRES_H
#define ATTNRES_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { ATTNRES_F32 = 0, ATTNRES_BF16 = 1 } attnres_dtype;

typedef enum {
  ATTNRES_OK = 0,
  ATTNRES_ERR_INVALID_ARG = 1,
  ATTNRES_ERR_UNSUPPORTED = 2,
  ATTNRES_ERR_CUDA = 3,
  ATTNRES_ERR_TIMEOUT = 4
} attnres_status;

/* Largest number of pseudo-queries one stage-1 call batches. */
#define ATTNRES_MAX_QUERIES 16

/*
 * attnres_full_fwd - one Full AttnRes read (DepthBench reading notes section
 * 2.3, paper Appendix A; LLMRes blog "Kimi AttnRes", h_l = sum_i alpha_{i->l} v_i).
 *
 *   V          device, [n_src, T, d] sources (slice i at V + i*src_stride
 *              elements), dtype v_dtype. Slice 0 is the embedding.
 *   src_stride elements between consecutive sources, >= T*d.
 *   n_src      number of sources, >= 1 (n_src == 1 returns v_0 exactly).
 *   w, gamma   device, fp32 [d]: the read's pseudo-query and key-RMSNorm gain.
 *   eps        RMSNorm epsilon, >= 0.
 *   out        device, [T, d] of out_dtype; must not overlap V.
 */
int attnres_full_fwd(const void* V, int64_t src_stride, int32_t n_src, int64_t T,
                     int32_t d, int32_t v_dtype, const float* w, const float* gamma,
                     float eps, void* out, int32_t out_dtype, void* stream);

/*
 * attnres_full_pass - R consecutive Full AttnRes reads over one stored
 * history: read r aggregates V[0 .. r] (r + 1 sources) with W[r], Gamma[r]
 * and writes out + r*out_stride. This is the read sequence of a Full AttnRes
 * model whose sublayer r's output is V[r + 1] (DepthBench reading notes
 * section 2.3: the first sublayer reads the embedding alone; with R = 2L + 1
 * the last read is the LM-head read).
 *
 *   V        device, [R, T, d] history, dtype v_dtype, src_stride >= T*d.
 *   W, Gamma device, fp32 [R, d].
 *   out      device, R outputs [T, d] of out_dtype, out_stride >= T*d
 *            elements apart; must not overlap V.
 */
int attnres_full_pass(const void* V, int64_t src_stride, int32_t R, int64_t T,
                      int32_t d, int32_t v_dtype, const float* W, const float* Gamma,
                      float eps, void* out, int64_t out_stride, int32_t out_dtype,
                      void* stream);

/*
 * attnres_full_fwd_prenorm / attnres_full_pass_prenorm - the same reads,
 * each also emitting the consuming sublayer's pre-norm of its result
 * (DepthBench reading notes section 2.3: the sublayer computes
 * f_l = F_l(RMSNorm_pre,l(z_l)) from the aggregated z_l). The row is
 * normalised while it is still in registers, which saves the sublayer a read
 * of z:
 *
 *   out_normed[t, k] = gamma_pre[k] * z[t, k] / sqrt(mean_k z[t, k]^2 + eps_pre)
 *
 * from z in fp32 before it is rounded to out_dtype.
 *
 *   gamma_pre   device, fp32 [d] (pass: [R, d], row r for read r).
 *   eps_pre     >= 0.
 *   out         as for the plain read, or NULL: z itself is then not stored.
 *   out_normed  device, [T, d] of out_dtype (pass: R of them, out_stride
 *               elements apart, like out); must not overlap V, out, W,
 *               Gamma or gamma_pre. Not NULL.
 */
int attnres_full_fwd_prenorm(const void* V, int64_t src_stride, int32_t n_src, int64_t T,
                             int32_t d, int32_t v_dtype, const float* w, const float* gamma,
                             float eps, const float* gamma_pre, float eps_pre, void* out,
                             void* out_normed, int32_t out_dtype, void* stream);
int attnres_full_pass_prenorm(const void* V, int64_t src_stride, int32_t R, int64_t T,
                              int32_t d, int32_t v_dtype, const float* W, const float* Gamma,
                              float eps, const float* Gamma_pre, float eps_pre, void* out,
                              void* out_normed, int64_t out_stride, int32_t out_dtype,
                              void* stream);

/*
 * attnres_query_projection / attnres_full_fwd_dynq - the input-dependent
 * query (the ablation the pages report: LLMRes blog, on the paper's ablation:
 * a query projected from the current hidden state by a per-layer d x d matrix
 * instead of the fixed learned pseudo-query).
 *
 * attnres_query_projection: Q[t, j] = sum_k Wq[j, k] H[t, k], i.e. Q = H Wq^T,
 * on the tensor cores (bf16 inputs, fp32 sums).
 *   H    device, [T, d] of h_dtype (ATTNRES_BF16 only; else UNSUPPORTED).
 *   Wq   device, bf16 [d, d], row j the weights of query feature j.
 *   Q    device, fp32 [T, d]; must not overlap H or Wq.
 *
 * attnres_full_fwd_dynq: the Full read with token t scored by its own query:
 * e_i(t) = Q[t] . (gamma * v_i(t)) / rms(v_i(t)); otherwise as
 * attnres_full_fwd (there is no shared w).
 *   Q    device, fp32 [T, d]; must not overlap out.
 */
int attnres_query_projection(const void* H, int64_t T, int32_t d, int32_t h_dtype, const void* Wq,
                             float* Q, void* stream);
int attnres_full_fwd_dynq(const void* V, int64_t src_stride, int32_t n_src, int64_t T, int32_t d,
                          int32_t v_dtype, const float* Q, const float* gamma, float eps, void* out,
                          int32_t out_dtype, void* stream);

/*
 * attnres_rmsnorm - RMSNorm of each row, out = gamma * x / sqrt(mean(x^2) + eps)
 * in fp32, stored in dtype: the sublayer pre-norm for a row no aggregation
 * call produces with it (the first sublayer of a block, whose output is
 * stage 1's O[0]).
 *
 *   x, out   device, [T, d] of dtype; out may be x (in place) but must not
 *            otherwise overlap it.
 *   gamma    device, fp32 [d].  eps >= 0.
 */
int attnres_rmsnorm(const void* x, int64_t T, int32_t d, int32_t dtype, const float* gamma,
                    float eps, void* out, void* stream);

/*
 * attnres_full_bwd - backward of one read over V[0 .. n_src): given
 * dz = dL/dz of its result, ADD the gradients with respect to the sources,
 * the query and the key-norm gain into dV, dw and dgamma. The read is
 * e_i = r_i (u . v_i), u = w * gamma, r_i = 1 / sqrt(mean_k v_ik^2 + eps),
 * a = softmax_i(e), z = sum_i a_i v_i (DepthBench reading notes section 2.3);
 * by the chain rule, per token:
 *   dL/da_i = dz . v_i,  dL/de_i = a_i (dL/da_i - sum_j a_j dL/da_j),
 *   dL/dv_i = a_i dz + dL/de_i (r_i u - e_i r_i^2 v_i / d),
 *   dL/du = sum over tokens and i of dL/de_i r_i v_i, dw = dL/du * gamma,
 *   dgamma = dL/du * w.
 * Accumulation (+=) lets a model's backward add every later read's share to
 * a source's gradient; zero the buffers before the first call.
 *
 *   V, src_stride, n_src, T, d, v_dtype, w, gamma, eps   as attnres_full_fwd.
 *   dz         device, [T, d] of dz_dtype.
 *   dV         device, fp32, n_src slices [T, d] dv_stride elements apart
 *              (>= T*d when n_src > 1); added to with atomic adds.
 *   dw, dgamma device, fp32 [d], added to; either may be NULL (skipped).
 * None of dV, dw, dgamma may overlap each other or an input. Returns
 * ATTNRES_ERR_UNSUPPORTED for shapes no kernel covers (d > 16384 off the
 * fast path). Results depend on the order of atomic additions only within
 * fp32 rounding.
 */
int attnres_full_bwd(const void* V, int64_t src_stride, int32_t n_src, int64_t T, int32_t d,
                     int32_t v_dtype, const float* w, const float* gamma, float eps,
                     const void* dz, int32_t dz_dtype, float* dV, int64_t dv_stride, float* dw,
                     float* dgamma, void* stream);

/*
 * attnres_block_bwd - gradients of a whole Block pass (the pass of
 * attnres_block_pass) with respect to the embedding, every sublayer output,
 * and every read's query and key gain, given dL/dout_k for every sublayer k.
 * Block AttnRes (DepthBench reading notes section 2.5; LLMRes blog, "Block
 * Attention Residuals"): sublayer k = n * S + j reads {embedding, b_1 .. b_n,
 * P_k if j >= 1}, with b_m the plain sum of block (m-1)'s outputs and P_k the
 * sum of block n's outputs before k. By the chain rule the gradient of b_m
 * reaches every member of block m-1 unchanged and that of P_k every output of
 * block n before k. All dL/dout_k are inputs (the vector-Jacobian product of
 * the pass with F given, as the forward defines it; a model whose sublayers
 * make F from the outputs runs the read backward per sublayer instead). For d
 * a multiple of 128 up to 1024, at most 8 blocks and 8 sublayers per block,
 * each block's S reads run in one batched pass over the tokens; otherwise the
 * reads run in reverse order through the Full read's backward over fp32
 * copies of their sources. Either way the running sums are rebuilt by the
 * same fp32 additions the forward made.
 *
 *   Src       device, [N][T][d] dtype, rows src_stride apart: Src[0] the
 *             embedding, Src[m] the frozen summary b_m (as the forward pass
 *             left them); row N (if any) is not read.
 *   F         device, [N*S][T][d] dtype: the sublayer outputs, f_stride apart.
 *   W, Gamma  device, fp32 [N*S][d]: each read's query and key gain.
 *   dOut      device, [N*S][T][d] dout_dtype: dL/dout_k, dout_stride apart.
 *   dEmb      device, fp32 [T][d], +=.
 *   dF        device, fp32 [N*S][T][d], +=, df_stride apart.
 *   dW, dGamma device, fp32 [N*S][d], +=; may be NULL.
 *   scratch   device, fp32, at least attnres_block_bwd_scratch_floats(N, S,
 *             T, d) floats (the caller's; contents on return unspecified).
 * Returns ATTNRES_ERR_INVALID_ARG for bad sizes, strides, a short scratch or
 * outputs overlapping inputs or each other; launch errors as ATTNRES_ERR_CUDA.
 */
int attnres_block_bwd(const void* Src, int64_t src_stride, const void* F, int64_t f_stride, int32_t N,
                      int32_t S, int64_t T, int32_t d, int32_t dtype, const float* W, const float* Gamma,
                      float eps, const void* dOut, int64_t dout_stride, int32_t dout_dtype, float* dEmb,
                      float* dF, int64_t df_stride, float* dW, float* dGamma, float* scratch,
                      int64_t scratch_floats, void* stream);
/* Scratch attnres_block_bwd needs: (2 (N + 1) + S + 1) * T * d floats; -1 for bad sizes. */
int64_t attnres_block_bwd_scratch_floats(int32_t N, int32_t S, int64_t T, int32_t d);

/*
 * attnres_block_stage1 - stage 1 of the two-stage Block AttnRes computation
 * (datacamp explainer, "two-stage computation"): the S pseudo-queries of one
 * block against the cross-block sources, each source row read once for all S.
 *
 *   Src        device, [n_src, T, d] cross-block sources (embedding, then the
 *              completed block sums), dtype, src_stride >= T*d.
 *   W, Gamma   device, fp32 [S, d], one row per sublayer of the block.
 *   S          1 <= S <= ATTNRES_MAX_QUERIES.
 *   O          host array of S device pointers; O[j] receives the normalised
 *              read of query j over Src, [T, d] of dtype. For the first
 *              sublayer of a block (empty running sum) O[0] is its final
 *              output. O[j] must not overlap Src or each other.
 *   lse        device, fp32 [S, T] (row j at lse + j*T): log sum_i exp(e_ij),
 *              the softmax mass stage 2 merges on. May be NULL (not written).
 */
int attnres_block_stage1(const void* Src, int64_t src_stride, int32_t n_src, int64_t T,
                         int32_t d, int32_t dtype, const float* W, const float* Gamma,
                         int32_t S, float eps, void* const* O, float* lse, void* stream);

/*
 * attnres_stage1_dsplit_partials / attnres_stage1_dsplit_finish - stage 1 with
 * the features split into shards (datacamp explainer, system optimisations,
 * "memory-efficient prefill": block representations sharded across
 * tensor-parallel devices; read as a feature split, where each device keeps a
 * slice of every source row and only score statistics cross devices). A score needs
 * ss = sum_k v_k^2 and dot_j = sum_k w_jk gamma_jk v_k over all d features;
 * both are sums, so each shard forms its part and the parts are added (the one
 * exchange step: an all-reduce of (1 + S) floats per (source, token)). With the
 * totals, each shard finishes the softmax and its own features of the outputs.
 *
 * partials:
 *   Src       device, [n_src, T, d_shard] the shard's features, src_stride >= T*d_shard.
 *   W, Gamma  device, fp32 [S, d_shard], the shard's slice of each query row.
 *   partials  device, fp32 [T][n_src][S + 1]: for token t and source i, entry 0
 *             holds ss, entry 1 + j dot_j. accumulate != 0 adds to it (the
 *             shards of one GPU in turn); 0 overwrites.
 * finish:
 *   Src       as above; d_total the full feature count (mean of squares).
 *   partials  the totals over all shards.
 *   O         host array of S device pointers, [T, d_shard] each: the shard's
 *             features of each query's normalised read.
 *   lse       device, fp32 [S, T] or NULL.
 * Kernels: bf16 shards whose width is a multiple of 64 stream the sources by
 * TMA and take the dots, sum v^2 and (with at most 16 sources) the weighted
 * sums on the tensor cores; other shapes take FMA kernels.
 * Shards wider than 512 features, or unaligned buffers, return
 * ATTNRES_ERR_UNSUPPORTED.
 */
int attnres_stage1_dsplit_partials(const void* Src, int64_t src_stride, int32_t n_src, int64_t T,
                                   int32_t d_shard, int32_t dtype, const float* W,
                                   const float* Gamma, int32_t S, float* partials,
                                   int32_t accumulate, void* stream);
int attnres_stage1_dsplit_finish(const void* Src, int64_t src_stride, int32_t n_src, int64_t T,
                                 int32_t d_shard, int32_t d_total, int32_t dtype,
                                 const float* partials, int32_t S, float eps, void* const* O,
                                 float* lse, void* stream);

/*
 * attnres_block_merge - stage 2 for one sublayer: extend the block's running
 * sum and merge it, as one more softmax source, with the stage-1 result
 * (datacamp explainer, "two-stage computation": online-softmax merge of the
 * intra-block dependency; DepthBench reading notes section 2.5: a read sees
 * the embedding, the frozen blocks and the current running sum).
 *
 *   O_j, lse_j device, stage-1 output [T, d] (dtype) and fp32 [T] of this query.
 *   P          device, fp32 [T, d] running sum, read and written in place.
 *   f_prev     device, [T, d] dtype, or NULL. Non-NULL: P <- P + f_prev first
 *              (P <- f_prev when p_is_empty != 0). NULL: P is used as it is
 *              and is not written; p_is_empty must then be 0.
 *   w, gamma   device, fp32 [d] of this sublayer.
 *   out        device, [T, d] dtype: the sublayer's aggregated input.
 *              out must not overlap O_j, P or f_prev.
 */
int attnres_block_merge(const void* O_j, const float* lse_j, float* P, const void* f_prev,
                        int32_t p_is_empty, const float* w, const float* gamma, float eps,
                        int64_t T, int32_t d, int32_t dtype, void* out, void* stream);

/*
 * attnres_block_merge_prenorm - the same merge, also emitting the sublayer's
 * pre-norm of the merged row (see attnres_full_fwd_prenorm):
 * out_normed = gamma_pre * z / sqrt(mean(z^2) + eps_pre) from z in fp32.
 * out may be NULL (z not stored); out_normed ([T, d] dtype, not NULL) must not
 * overlap out, O_j, lse_j, P or f_prev.
 */
int attnres_block_merge_prenorm(const void* O_j, const float* lse_j, float* P,
                                const void* f_prev, int32_t p_is_empty, const float* w,
                                const float* gamma, float eps, const float* gamma_pre,
                                float eps_pre, int64_t T, int32_t d, int32_t dtype, void* out,
                                void* out_normed, void* stream);

/*
 * attnres_block_summary_accumulate - running sum of a block and the block
 * summary (LLMRes blog "Block Attention Residuals": a block is represented by
 * the sum of its sublayer outputs; datacamp explainer: b_n = sum of the
 * outputs of the layers in block n, with b_0 the embedding).
 *
 *   P            device, fp32 [T, d] running sum.
 *   f            device, [T, d] dtype: a sublayer output to add.
 *   p_is_empty   non-zero: the running sum is empty (treated as 0, P not read).
 *   summary_out  NULL: accumulate, P <- P + f.
 *                non-NULL: freeze, summary_out <- P + f rounded to dtype
 *                ([T, d] dtype, device); P is then not written.
 */
int attnres_block_summary_accumulate(float* P, const void* f, int32_t p_is_empty,
                                     void* summary_out, int64_t T, int32_t d, int32_t dtype,
                                     void* stream);

/*
 * attnres_block_merge_parts - the stage-2 merge with the running sum given in
 * parts: P_j = P_base + f_0 + ... + f_{n_parts-1}, the sum of the block's
 * first j outputs (LLMRes blog "Block Attention Residuals": the running sum
 * of the current block is one more softmax source, DepthBench reading notes
 * section 2.5), formed in fp32 and added in that order. This is the order in
 * which the one-step calls above build it, so keeping a sum in P or forming
 * it again from the outputs gives the same bits. Re-reading a few bf16
 * outputs moves fewer bytes than storing and reloading an fp32 sum; the Block
 * pass chooses by attnres_block_running_sum_plan.
 *
 *   O_j, lse_j  as in attnres_block_merge.
 *   P_base      device, fp32 [T, d]: a stored running sum to start from, or
 *               NULL (the sum starts from the first part; n_parts >= 1).
 *   F_parts     device, the n_parts outputs [T, d] dtype, part_stride >= T*d
 *               elements apart (part_stride unused when n_parts <= 1); n_parts
 *               from 0 (P_base used as it is) to 16.
 *   P_out       device, fp32 [T, d], or NULL: where P_j is stored. It may be
 *               P_base itself (in place) but must not overlap anything else.
 *   w, gamma    device, fp32 [d] of this sublayer.
 *   out         device, [T, d] dtype; overlaps no other argument.
 *   summary_out device, [T, d] dtype, or NULL. When given, F_parts holds one
 *               output more (n_parts + 1 of them, at most 16) and summary_out
 *               receives P_j + f_{n_parts}, added in fp32 after the others
 *               and rounded: the block's summary, frozen by its last merge
 *               (the same bits as attnres_block_summary_parts over all
 *               n_parts + 1 parts). Overlaps no other argument.
 * Errors as attnres_block_merge.
 */
int attnres_block_merge_parts(const void* O_j, const float* lse_j, const float* P_base,
                              const void* F_parts, int64_t part_stride, int32_t n_parts,
                              float* P_out, const float* w, const float* gamma, float eps,
                              int64_t T, int32_t d, int32_t dtype, void* out, void* summary_out,
                              void* stream);

/*
 * attnres_block_summary_parts - a running sum from parts (as in
 * attnres_block_merge_parts, n_parts from 1 to 16): summary_out <- P_base +
 * f_0 + ... rounded to dtype (the freeze of a block summary), or, with
 * summary_out NULL, P_out <- that sum in fp32 (P_out may be P_base).
 */
int attnres_block_summary_parts(const float* P_base, const void* F_parts, int64_t part_stride,
                                int32_t n_parts, float* P_out, void* summary_out, int64_t T,
                                int32_t d, int32_t dtype, void* stream);

/*
 * attnres_block_running_sum_plan - which running sums attnres_block_pass keeps
 * in P_scratch for blocks of S sublayers stored as dtype: stored[j] = 1 for
 * each 1 <= j < S whose P_j is written (stored[0] = stored[S] = 0). Every
 * other P_j is formed from the last kept one, or from nothing, plus the
 * outputs since; the plan minimises the bytes each element moves (an output
 * re-read costs 2 or 4 bytes, a kept fp32 sum 4 to write and 4 to read).
 * Example: bf16, S = 6 keeps P_4 only. stored has S + 1 entries (host).
 */
int attnres_block_running_sum_plan(int32_t S, int32_t dtype, int32_t* stored);

/*
 * attnres_block_pass - the reads of N blocks of S sublayers by the two-stage
 * computation, for stored sublayer outputs F (the synthetic sequencing a
 * model would interleave with its sublayers). Block n (0-based) runs stage 1
 * over Src[0 .. n], S - 1 merges and, unless it is the last block and
 * freeze_last == 0, freezes its summary into Src[n + 1].
 *
 *   F           device, [N*S, T, d] sublayer outputs, dtype, f_stride >= T*d.
 *   W, Gamma    device, fp32 [N*S, d].
 *   Src         device, [N + freeze_last, T, d] dtype, src_stride >= T*d.
 *               Src[0] holds the embedding (input); Src[1 ..] are written.
 *   O_scratch   device, [max(S-1,1), T, d] dtype workspace (stage-1 results).
 *   lse_scratch device, fp32 [S, T] workspace.
 *   P_scratch   device, fp32 [T, d] workspace (the running sums that
 *               attnres_block_running_sum_plan says to keep).
 *   out         device, N*S outputs [T, d] dtype, out_stride >= T*d apart.
 * Merge j of a block takes its running sum as the last kept one plus the
 * outputs since (attnres_block_merge_parts); the freeze likewise
 * (attnres_block_summary_parts).
 */
int attnres_block_pass(const void* F, int64_t f_stride, int32_t N, int32_t S, int64_t T,
                       int32_t d, int32_t dtype, const float* W, const float* Gamma,
                       float eps, void* Src, int64_t src_stride, int32_t freeze_last,
                       void* O_scratch, float* lse_scratch, float* P_scratch,
                       void* out, int64_t out_stride, void* stream);

/*
 * attnres_block_pass_noalloc - attnres_block_pass for callers that cannot
 * allocate device memory. (The pages have no counterpart: this is a library
 * convenience, not part of the method.)
 *
 * Some callers have no device memory to lend as workspace and may not call
 * cudaMalloc: a serving process that reserves and budgets all device memory
 * up front and forbids allocation afterwards, or a caller running on a thread
 * that must never make a call that can implicitly synchronise the device,
 * which cudaMalloc and cudaFree can do. This entry point takes the same
 * inputs and outputs as attnres_block_pass (F, W, Gamma, Src, out) but no
 * workspace: the stage-1 results, their log-masses and the fp32 running sum
 * live in one array of ATTNRES_NOALLOC_SCRATCH_BYTES bytes that the library
 * defines at file scope. It calls no cudaMalloc, cudaFree or other
 * allocating routine.
 *
 *   - Size limit: the workspace of a call needs
 *     (S > 1 ? (S-1)*T*d*es + 4*T*d : 0) + 4*S*T bytes (es = 2 for bf16, 4
 *     for fp32; each part rounded up to 256 bytes). A call that needs more
 *     than ATTNRES_NOALLOC_SCRATCH_BYTES returns ATTNRES_ERR_UNSUPPORTED and
 *     launches nothing. Example: bf16, d = 1024, S = 8 fits up to T = 3634.
 *     The pointer, dtype, eps and stride checks come first, so a call that is
 *     both malformed and too large returns ATTNRES_ERR_INVALID_ARG (except
 *     when T or d alone exceeds the array's size: ATTNRES_ERR_UNSUPPORTED).
 *   - Memory: every CUDA context that loads the library's device code holds
 *     the array (64 MiB) until the context is destroyed or the process
 *     exits. With lazy module loading (the CUDA default) the array is
 *     allocated when this entry point first runs in a context, and that first
 *     call may synchronise the device while the module loads; with
 *     CUDA_MODULE_LOADING=EAGER it is allocated when the context is created,
 *     in every process that loads the library. A caller that budgets device
 *     memory up front, or that must not synchronise later, should therefore
 *     make one small warm-up call (for example T = 1) at start-up, before it
 *     reserves its memory or starts its no-sync thread.
 *   - Set-up: the first call in a CUDA context, with that context current,
 *     looks up the array's device address (cudaGetSymbolAddress) and caches
 *     it under the context's id. Make that first call before any stream
 *     capture begins. After cudaDeviceReset, or when a primary context is
 *     released and created again, the array is a new one: the next call looks
 *     its address up again (and is then such a first call).
 *   - Sharing: all calls in a context share the one array, and it keeps the
 *     contents of the last call. Nothing in it needs to start at zero (every
 *     byte a call reads was written earlier in the same call). Calls whose
 *     work overlaps on the GPU (for example on two streams) race on the
 *     array: order them on one stream or with events.
 *   - Otherwise as attnres_block_pass (same arguments, checks and statuses).
 */
#define ATTNRES_NOALLOC_SCRATCH_BYTES (64ull * 1024ull * 1024ull)
int attnres_block_pass_noalloc(const void* F, int64_t f_stride, int32_t N, int32_t S, int64_t T,
                               int32_t d, int32_t dtype, const float* W, const float* Gamma,
                               float eps, void* Src, int64_t src_stride, int32_t freeze_last,
                               void* out, int64_t out_stride, void* stream);

/*
 * attnres_device_status - synchronise `stream` and report device-side
 * failures of earlier calls on the current device: ATTNRES_ERR_TIMEOUT if a
 * kernel gave up a bounded wait since the last call (the record is then
 * cleared), ATTNRES_ERR_CUDA on a pending CUDA error, else ATTNRES_OK.
 */
int attnres_device_status(void* stream);

/*
 * attnres_selftest_wait_timeout - checks the bounded-wait failure path on the
 * current device: launches one CTA whose mbarrier wait is never satisfied (no
 * thread arrives and no copy is issued), so the wait runs out after its limit
 * (about 2 s), records a timeout and returns. A following
 * attnres_device_status(stream) reports ATTNRES_ERR_TIMEOUT and clears the
 * record; the context stays usable. Returns the launch status.
 */
int attnres_selftest_wait_timeout(void* stream);

/*
 * Failure-path test hooks. The pages define no error handling; these exist so
 * that tests can drive the library's error paths without faulting a GPU. Both
 * are off by default, process-wide (all devices and threads), and meant for
 * tests only.
 *
 * attnres_test_fail_launch - arms a simulated launch failure: after `after`
 * more launches succeed (kernels, and the memsets and copies of the Block
 * backward), the next launch is not made and its call returns
 * ATTNRES_ERR_CUDA, as a real launch error would; the hook then disarms
 * itself. A call that makes several launches (a Full or Block pass) stops at
 * the failed one: the launches before it ran, nothing after it is enqueued.
 * after < 0 disarms. Returns the previous setting (-1 once an armed failure
 * has fired), so a test can tell whether it was consumed.
 */
int64_t attnres_test_fail_launch(int64_t after);

/*
 * attnres_test_withhold_stage - makes the copy producer of one pipelined
 * kernel leave one stage unfilled, so the consumers' bounded wait for it runs
 * out (after about 2 s): the kernel records a timeout and returns, and
 * attnres_device_status reports ATTNRES_ERR_TIMEOUT. kernel: 0 = off, 1 = the
 * Full-read bulk kernel (index counts the (tile, source) copies of each CTA),
 * 2 = the tensor-core stage 1 (index counts each CTA's tiles), 3 = the tiled
 * merge (index counts each CTA's tiles; tiles fetched before the previous
 * kernel finishes, in a Block pass, are never withheld). Every CTA with more
 * than `index` copies withholds its copy number `index`; its other copies are
 * issued and waited for before the CTA exits. Stays set until changed.
 * Returns ATTNRES_ERR_INVALID_ARG for an unknown kernel or a negative index.
 */
int attnres_test_withhold_stage(int32_t kernel, int64_t index);

/* Static description of a status code (never NULL). */
const char* attnres_status_string(int32_t status);

/*
 * attnres_kernel_path - which kernel a call with these arguments would use:
 * 1 = the fast kernel, 0 = the general kernel, negative = invalid arguments.
 * op: 0 full read, 1 stage 1, 2 merge, 3 accumulate, 4 query projection
 * (attnres_query_projection with H = Wq = src and Q = out; dtype must be
 * ATTNRES_BF16): 2 = tensor-core tiles shared by pairs of CTAs, 1 = tensor-core
 * tiles of one CTA, 0 = another kernel. Pointers are only inspected for
 * alignment; n_or_s is n_src for op 0 and 1, ignored otherwise; s is S for
 * op 1. Op 4 asks the device how many CTA pairs fit, so it wants one.
 */
int attnres_kernel_path(int32_t op, const void* src, const void* out, int32_t n_or_s,
                        int32_t s, int64_t T, int32_t d, int32_t dtype);

/* ABI version of this header: 1. */
int attnres_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* ATTNRES_H */
