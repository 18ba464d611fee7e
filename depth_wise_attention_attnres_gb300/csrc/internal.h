// Internal launcher interface between the C ABI layer and the kernel files.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "attnres.h"

namespace attnres {

// One Full AttnRes read (one query) over n_src sources.
// The consuming sublayer's pre-norm, emitted next to an aggregated row z:
// out = gamma * z / sqrt(mean(z^2) + eps), from z in fp32 before rounding
// (DepthBench reading notes section 2.3: f_l = F_l(RMSNorm_pre,l(z_l))).
struct PreNorm {
  const float* gamma;   // [d]; nullptr: no pre-norm output
  float eps;
  void* out;            // [T, d] in the output dtype
};

struct FullArgs {
  const void* V;
  int64_t src_stride;  // elements
  int n_src;
  int64_t T;
  int d;
  int v_bf16;
  const float* w;
  const float* gamma;
  float eps;
  void* out;
  int out_bf16;
  // Reads of one pass after the first: none of their inputs is written by the
  // read before them, so they wait for it (griddepcontrol.wait) at their end
  // instead of their start, which keeps the reads completing in order while a
  // read's loads overlap the tail of the previous one.
  int late_wait;
  PreNorm pre;          // out may be nullptr when pre.gamma is set
  const float* Q;       // [T, d] fp32 per-token query (input-dependent); w then unused
  // Failure-path test hook (attnres_test_withhold_stage): the producer of each
  // CTA leaves its copy number `withhold` unissued, so the consumers' bounded
  // wait for it runs out. -1 (the default) withholds nothing.
  int64_t withhold = -1;
};

// S queries over the same n_src sources (stage 1; the general kernel also
// serves a single Full read with S = 1).
struct MultiArgs {
  const void* V;
  int64_t src_stride;
  int n_src;
  int64_t T;
  int d;
  int bf16;             // storage dtype of V and of every output
  const float* W;       // [S, d]
  const float* Gamma;   // [S, d]
  int S;
  float eps;
  void* out[ATTNRES_MAX_QUERIES];
  float* lse;           // [S, T] or nullptr
  PreNorm pre;          // S == 1 only (a Full read); out[0] may then be nullptr
  const float* Q;       // S == 1 only: [T, d] fp32 per-token query instead of W
  int64_t withhold = -1;  // test hook of the tensor-core stage 1 (as FullArgs)
};

// Stage-2 merge of one sublayer (merge.cu). The running sum it merges is
// formed as base + f_0 + ... + f_{q-1}, added in that order in fp32 (the
// order the forward's sequential running sum uses, so any split between a
// stored base and re-read outputs gives the same bits).
struct MergeArgs {
  const void* O;
  const float* lse;
  const float* P;       // stored fp32 running sum to start from; nullptr: none
  const void* parts;    // the q sublayer outputs added to it, part_stride apart
  int64_t part_stride;  // elements
  int nparts;           // q >= 0; q == 0 needs P
  float* P_out;         // the resulting running sum (fp32, may be P); nullptr: not stored
  const float* w;
  const float* gamma;
  float eps;
  int64_t T;
  int d;
  int bf16;
  void* out;            // may be nullptr when pre.gamma is set
  PreNorm pre;
  // Fetch the first tiles of O_j and the parts before waiting for the previous
  // kernel: only when that kernel writes none of them (in a Block pass, the
  // merge before). 2: the parts only (after stage 1, which writes O_j).
  int early;
  int64_t withhold = -1;  // test hook of the tiled merge (as FullArgs)
  // Also store round(running sum + parts[nparts]) here:
  // a block's summary, the freeze fused into its last merge. nullptr: none.
  void* summary = nullptr;
};
constexpr int kMaxMergeParts = 16;

// Backward of one read (full_bwd.cu): dV, dw, dgamma accumulated in fp32.
struct BwdArgs {
  const void* V;
  int64_t src_stride;   // elements
  int n_src;
  int64_t T;
  int d;
  int v_bf16;
  const float* w;
  const float* gamma;
  float eps;
  const void* dz;       // dL/dz [T, d]
  int dz_bf16;
  float* dV;            // [n_src, T, d] fp32, += ; sources dv_stride elements apart
  int64_t dv_stride;
  float* dw;            // [d] fp32, += ; may be nullptr
  float* dgamma;        // [d] fp32, += ; may be nullptr
};
constexpr int kMaxBwdFastSources = 256;   // per-(row, source) scalars live in shared memory
constexpr int kMaxBwdGenericD = 16384;    // du of a CTA lives in shared memory

// Block stage 1 over one feature shard (dsplit.cu).
struct DsplitArgs {
  const void* Src;      // [n_src, T, d_shard] the shard's features of each source
  int64_t src_stride;   // elements
  int n_src;
  int64_t T;
  int d_shard;
  int d_total;          // the full width (the mean of squares divides by it)
  int bf16;
  const float* W;       // [S, d_shard] the shard's slice of each query
  const float* Gamma;   // [S, d_shard]
  int S;
  float eps;
  float* partials;      // [T][n_src][S + 1] fp32: sum v^2, then the S dots
  int accumulate;       // partials: add to the buffer instead of writing it
  void* out[ATTNRES_MAX_QUERIES];  // finish: [T, d_shard] per query
  float* lse;           // finish: [S, T] or nullptr
};
constexpr int kMaxDsplitShard = 512;

// Running-sum update or freeze (merge.cu): base + f_0 + ... + f_{q-1} in
// fp32, in that order, into P_out (fp32) or, rounded, into summary.
struct AccumArgs {
  const float* P;       // base; nullptr: none
  const void* parts;    // q >= 1 sublayer outputs, part_stride apart
  int64_t part_stride;
  int nparts;
  float* P_out;         // fp32 result (may be P); used when summary is nullptr
  void* summary;        // storage-dtype result; nullptr: write P_out
  int64_t T;
  int d;
  int bf16;
  // Skip the wait for the previous kernel: only when no kernel that may still
  // be running writes what this one reads or reads what it writes (in a Block
  // pass, the freeze after the block's last merge).
  int no_wait = 0;
};

// Kernel selection (pure functions of the arguments).
bool full_fast_ok(const FullArgs& a);
bool stage1_fast_ok(const MultiArgs& a);
bool stage1_tc_ok(const MultiArgs& a);
bool merge_fast_ok(const MergeArgs& a);
bool accum_fast_ok(const AccumArgs& a);

// Launchers: enqueue on `s` and return the launch's CUDA error.
cudaError_t launch_full_fast(const FullArgs& a, cudaStream_t s);
cudaError_t launch_multi_generic(const MultiArgs& a, cudaStream_t s);
cudaError_t launch_stage1_fast(const MultiArgs& a, cudaStream_t s);
cudaError_t launch_stage1_tc(const MultiArgs& a, cudaStream_t s);
cudaError_t launch_merge(const MergeArgs& a, cudaStream_t s, bool fast);
cudaError_t launch_accum(const AccumArgs& a, cudaStream_t s, bool fast);
// RMSNorm of each row of x [T, d] (storage dtype in and out; out may be x).
cudaError_t launch_rmsnorm(const void* x, int64_t T, int d, int is_bf16, const float* gamma, float eps, void* out,
                           cudaStream_t s);
cudaError_t launch_wait_timeout_selftest(cudaStream_t s);
bool full_bwd_fast_ok(const BwdArgs& a);
// Q = H Wq^T (bf16 H [T, d], Wq [d, d]; fp32 Q): the input-dependent query.
bool proj_ok(const void* H, const void* Wq, const float* Q, int d);
cudaError_t launch_proj(const void* H, const void* Wq, float* Q, int64_t T, int d, cudaStream_t s);
cudaError_t launch_proj_generic(const void* H, const void* Wq, float* Q, int64_t T, int d, cudaStream_t s);
bool proj_tc_ok(const void* H, const void* Wq, const float* Q, int64_t T, int d);
cudaError_t launch_proj_tensor(const void* H, const void* Wq, float* Q, int64_t T, int d, cudaStream_t s);
// 2: tcgen05 CTA pairs, 1: tcgen05 single CTAs, 0: neither (mma.sync or plain).
int proj_path(const void* H, const void* Wq, const float* Q, int64_t T, int d);
cudaError_t take_timeout_proj(unsigned int* flag);
bool dsplit_ok(const DsplitArgs& a);
cudaError_t launch_dsplit_partials(const DsplitArgs& a, cudaStream_t s);
cudaError_t launch_dsplit_finish(const DsplitArgs& a, cudaStream_t s);
cudaError_t take_timeout_dsplit(unsigned int* flag);
cudaError_t take_timeout_blockbwd(unsigned int* flag);
// The driver's cuTensorMapEncodeTiled, looked up once (nullptr if the driver
// lacks it).
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encode_fn();
cudaError_t launch_full_bwd(const BwdArgs& a, cudaStream_t s, bool fast);
// One block's reads in the batched Block backward (block_bwd.cu).
struct BlockBwdArgs {
  const void* Src;      // [N][T][d] embedding and frozen summaries
  int64_t src_stride;
  const void* F;        // sublayer outputs, f_stride apart
  int64_t f_stride;
  const float* W;       // [N*S][d]
  const float* Gamma;
  const void* dOut;     // dL/dout, dout_stride apart
  int64_t dout_stride;
  int dz_bf16;
  float* dVs;           // [N][E] gradients of the embedding and the summaries (+=)
  int64_t E;
  float* dF;            // df_stride apart (+=)
  int64_t df_stride;
  float* dW;            // may be nullptr
  float* dGamma;        // may be nullptr
  int N, S, n;          // n: the block
  int64_t T;
  int d;
  int bf16;
  float eps;
};
bool block_bwd_batched_ok(const BlockBwdArgs& a);
cudaError_t launch_block_bwd_batched(const BlockBwdArgs& a, cudaStream_t s);
// Block pass backward helpers (block_bwd.cu); E elements per row, fp32 rows E apart.
cudaError_t launch_widen_rows(const void* src, int64_t src_stride, int is_bf16, float* dst, int R, int64_t E,
                              cudaStream_t s);
cudaError_t launch_psum(float* dst, const float* prev, const void* f, int is_bf16, int64_t E, cudaStream_t s);
cudaError_t launch_gupdate(float* G, float* ds, float* dfp, int64_t E, cudaStream_t s);
cudaError_t launch_spread(float* dst, int64_t dst_stride, int R, const float* g, int64_t E, cudaStream_t s);
cudaError_t take_timeout_bwd(unsigned int* flag);

// Failure-path test hooks (api.cu), off by default. Which producer, if any,
// withholds a copy: the tile index to leave unissued, or -1.
enum WithholdKernel { kWithholdNone = 0, kWithholdFull = 1, kWithholdStage1Tc = 2, kWithholdMerge = 3 };
int64_t withhold_for(WithholdKernel k);

// Device-side timeout records of each kernel file: read and clear (blocking).
cudaError_t take_timeout_full(unsigned int* flag);
cudaError_t take_timeout_stage1(unsigned int* flag);
cudaError_t take_timeout_merge(unsigned int* flag);
cudaError_t take_timeout_stage1tc(unsigned int* flag);

// Shared launch helpers (api.cu).
int sm_count();
cudaError_t allow_dynamic_smem(const void* kernel, int bytes);
int blocks_per_sm(const void* kernel, int threads, int smem_bytes);

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Launch with programmatic stream serialization (see pdl_wait in common.cuh).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), unsigned grid, unsigned block, int smem,
                       cudaStream_t s, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = static_cast<size_t>(smem);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

}  // namespace attnres
