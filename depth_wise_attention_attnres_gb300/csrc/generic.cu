// General AttnRes read kernel: S queries over n sources, any d, any alignment.
//
// One warp per token row. Pass 1 scores every source for every query (lanes
// stride over d; two warp sums per source and query) and keeps the scores in
// shared memory; the softmax over depth turns them into weights and lse; pass
// 2 forms each output element as the weighted sum over sources. It serves
// shapes the fast kernels do not cover (tiny brute-force shapes, d not a
// multiple of the vector width, unaligned pointers) with the same arithmetic
// (fp32, RMSNorm on keys only, no 1/sqrt(d); DepthBench reading notes section
// 2.3).
#include <math.h>

#include "common.cuh"
#include "internal.h"

namespace attnres {
namespace {

constexpr int kWarpsPerBlock = 8;

template <typename T>
__device__ __forceinline__ float ld(const void* base, int64_t idx) {
  return to_f32(static_cast<const T*>(base)[idx]);
}

template <typename T>
__global__ void __launch_bounds__(kWarpsPerBlock * 32) multi_generic_kernel(MultiArgs a, int warps) {
  extern __shared__ float sc[];  // [warps][S][n] scores, then weights
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (warp >= warps) return;
  const int n = a.n_src, S = a.S, d = a.d;
  float* my = sc + static_cast<size_t>(warp) * S * n;
  const float inv_d = 1.0f / static_cast<float>(d);

  for (int64_t row = static_cast<int64_t>(blockIdx.x) * warps + warp; row < a.T;
       row += static_cast<int64_t>(gridDim.x) * warps) {
    // Pass 1: scores e_ij = w_j . (gamma_j * v_i) / rms(v_i).
    for (int i = 0; i < n; ++i) {
      const int64_t base = i * a.src_stride + row * d;
      float ss = 0.f;
      float dot[ATTNRES_MAX_QUERIES];
#pragma unroll
      for (int j = 0; j < ATTNRES_MAX_QUERIES; ++j) dot[j] = 0.f;
      for (int k = lane; k < d; k += 32) {
        const float x = ld<T>(a.V, base + k);
        ss += x * x;
#pragma unroll
        for (int j = 0; j < ATTNRES_MAX_QUERIES; ++j)
          if (j < S) {
            const float q = a.Q ? a.Q[row * d + k] : a.W[j * static_cast<int64_t>(d) + k];
            dot[j] += q * a.Gamma[j * static_cast<int64_t>(d) + k] * x;
          }
      }
      ss = warp_sum(ss);
      const float r = rsqrtf(ss * inv_d + a.eps);
#pragma unroll
      for (int j = 0; j < ATTNRES_MAX_QUERIES; ++j)
        if (j < S) {
          const float dj = warp_sum(dot[j]);
          if (lane == 0) my[j * n + i] = dj * r;
        }
    }
    __syncwarp();
    // Softmax over depth, one lane per query.
    if (lane < S) {
      float* e = my + lane * n;
      float m = e[0];
      for (int i = 1; i < n; ++i) m = fmaxf(m, e[i]);
      float z = 0.f;
      for (int i = 0; i < n; ++i) z += expf(e[i] - m);
      const float inv = 1.0f / z;
      for (int i = 0; i < n; ++i) e[i] = expf(e[i] - m) * inv;
      if (a.lse) a.lse[lane * a.T + row] = m + logf(z);
    }
    __syncwarp();
    // Pass 2: weighted sum of the raw values.
    for (int j = 0; j < S; ++j) {
      const float* p = my + j * n;
      float q = 0.f;
      for (int k = lane; k < d; k += 32) {
        float acc = 0.f;
        for (int i = 0; i < n; ++i) acc += p[i] * ld<T>(a.V, i * a.src_stride + row * d + k);
        if (a.out[j]) static_cast<T*>(a.out[j])[row * d + k] = from_f32<T>(acc);
        q = fmaf(acc, acc, q);
      }
      if (j == 0 && a.pre.gamma) {
        // Pass 3 (a Full read with the sublayer's pre-norm): the row again,
        // scaled by 1 / rms of its fp32 values.
        const float rr = rsqrtf(warp_sum(q) * inv_d + a.pre.eps);
        for (int k = lane; k < d; k += 32) {
          float acc = 0.f;
          for (int i = 0; i < n; ++i) acc += p[i] * ld<T>(a.V, i * a.src_stride + row * d + k);
          static_cast<T*>(a.pre.out)[row * d + k] = from_f32<T>(a.pre.gamma[k] * (acc * rr));
        }
      }
    }
    __syncwarp();
  }
}

}  // namespace

cudaError_t launch_multi_generic(const MultiArgs& a, cudaStream_t s) {
  const int per_warp = a.S * a.n_src * static_cast<int>(sizeof(float));
  int warps = kWarpsPerBlock;
  const int limit = 200 * 1024;
  while (warps > 1 && warps * per_warp > limit) --warps;
  if (static_cast<int64_t>(warps) * per_warp > limit) return cudaErrorInvalidValue;
  const int smem = warps * per_warp;
  const void* fn = a.bf16 ? reinterpret_cast<const void*>(&multi_generic_kernel<bf16>)
                          : reinterpret_cast<const void*>(&multi_generic_kernel<float>);
  cudaError_t e = allow_dynamic_smem(fn, smem);
  if (e != cudaSuccess) return e;
  int64_t blocks = (a.T + warps - 1) / warps;
  const int64_t cap = static_cast<int64_t>(sm_count()) * 8;
  if (blocks > cap) blocks = cap;
  if (a.bf16)
    multi_generic_kernel<bf16><<<static_cast<unsigned>(blocks), kWarpsPerBlock * 32, smem, s>>>(a, warps);
  else
    multi_generic_kernel<float><<<static_cast<unsigned>(blocks), kWarpsPerBlock * 32, smem, s>>>(a, warps);
  return cudaGetLastError();
}

}  // namespace attnres
