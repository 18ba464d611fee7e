// Block AttnRes stage 2 (online-softmax merge) and running-sum kernels.
//
// Merge, per token row (datacamp explainer, "two-stage computation"; the
// running sum of the current block is one more softmax source, DepthBench
// reading notes section 2.5):
//   P   <- P + f_prev                       (fp32 running sum, optional)
//   s_P  = w^T (gamma * P / sqrt(mean(P^2) + eps))
//   M    = max(lse, s_P),  a = exp(lse - M),  b = exp(s_P - M)
//   out  = (a * O + b * P) / (a + b)
// where (O, lse) is the stage-1 read of this sublayer over the cross-block
// sources. Accumulate / freeze (LLMRes blog "Block Attention Residuals": a
// block is represented by the sum of its outputs): P <- P + f, or
// summary <- round(P + f).
//
// Both are HBM-bound streaming kernels (a few flops per byte). The fast merge
// gives each thread one 16-byte chunk of a row (8 bf16 or 4 fp32 features),
// reduces the two row sums over the row's warps through shared memory and
// writes P and out with 16-byte stores.
#include <math.h>

#include "common.cuh"
#include "internal.h"

namespace attnres {
namespace {

constexpr int kBlock = 256;
constexpr int kWarps = kBlock / 32;

// ------------------------------------------------------------- fast merge --

template <typename T>
struct Chunk;
template <>
struct Chunk<bf16> {
  static constexpr int N = 8;
  __device__ static void load(const void* p, float (&x)[8]) {
    const uint4 v = *reinterpret_cast<const uint4*>(p);
    x[0] = bf16_lo(v.x); x[1] = bf16_hi(v.x); x[2] = bf16_lo(v.y); x[3] = bf16_hi(v.y);
    x[4] = bf16_lo(v.z); x[5] = bf16_hi(v.z); x[6] = bf16_lo(v.w); x[7] = bf16_hi(v.w);
  }
  __device__ static void store(void* p, const float (&x)[8]) {
    *reinterpret_cast<uint4*>(p) = make_uint4(pack_bf16x2(x[0], x[1]), pack_bf16x2(x[2], x[3]),
                                              pack_bf16x2(x[4], x[5]), pack_bf16x2(x[6], x[7]));
  }
};
template <>
struct Chunk<float> {
  static constexpr int N = 4;
  __device__ static void load(const void* p, float (&x)[4]) {
    const float4 v = *reinterpret_cast<const float4*>(p);
    x[0] = v.x; x[1] = v.y; x[2] = v.z; x[3] = v.w;
  }
  __device__ static void store(void* p, const float (&x)[4]) {
    *reinterpret_cast<float4*>(p) = make_float4(x[0], x[1], x[2], x[3]);
  }
};

template <int N>
__device__ __forceinline__ void load_f32(const float* p, float (&x)[N]) {
#pragma unroll
  for (int q = 0; q < N; q += 4) {
    const float4 v = *reinterpret_cast<const float4*>(p + q);
    x[q] = v.x; x[q + 1] = v.y; x[q + 2] = v.z; x[q + 3] = v.w;
  }
}
template <int N>
__device__ __forceinline__ void store_f32(float* p, const float (&x)[N]) {
#pragma unroll
  for (int q = 0; q < N; q += 4) *reinterpret_cast<float4*>(p + q) = make_float4(x[q], x[q + 1], x[q + 2], x[q + 3]);
}

// wpr: warps per row (power of two, <= 8). A block iteration covers
// kRows * (8 / wpr) rows; each thread handles one 16-byte chunk in kRows rows,
// so all their loads are in flight before the reduction barrier.
constexpr int kRows = 2;

template <typename T>
__global__ void __launch_bounds__(kBlock) merge_fast_kernel(MergeArgs a, int wpr) {
  constexpr int N = Chunk<T>::N;
  __shared__ float red[2][kRows][kWarps][2];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rpb = kWarps / wpr;
  const int slot = warp / wpr;
  const int wr = warp - slot * wpr;
  const int d = a.d;
  const int nchunk = d / N;
  const int c = wr * 32 + lane;
  const bool active = c < nchunk;
  const int k = c * N;

  pdl_trigger();
  pdl_wait();
  float wq[N];
  if (active) {
#pragma unroll
    for (int q = 0; q < N; ++q) wq[q] = a.w[k + q] * a.gamma[k + q];
  }
  const float inv_d = 1.0f / static_cast<float>(d);
  int par = 0;
  const int64_t step = static_cast<int64_t>(gridDim.x) * rpb * kRows;
  for (int64_t base = static_cast<int64_t>(blockIdx.x) * rpb * kRows; base < a.T; base += step, par ^= 1) {
    float p[kRows][N], o[kRows][N];
    bool live[kRows];
#pragma unroll
    for (int r = 0; r < kRows; ++r) {
      const int64_t row = base + r * rpb + slot;
      live[r] = active && row < a.T;
      if (live[r]) {
        const int64_t off = row * d + k;
        Chunk<T>::load(static_cast<const T*>(a.O) + off, o[r]);
        if (a.f) {
          float f[N];
          Chunk<T>::load(static_cast<const T*>(a.f) + off, f);
          if (a.p_empty) {
#pragma unroll
            for (int q = 0; q < N; ++q) p[r][q] = f[q];
          } else {
            load_f32<N>(a.P + off, p[r]);
#pragma unroll
            for (int q = 0; q < N; ++q) p[r][q] += f[q];
          }
        } else {
          load_f32<N>(a.P + off, p[r]);
        }
      }
    }
#pragma unroll
    for (int r = 0; r < kRows; ++r) {
      float ss = 0.f, dot = 0.f;
      if (live[r]) {
        const int64_t off = (base + r * rpb + slot) * d + k;
        if (a.f) store_f32<N>(a.P + off, p[r]);
#pragma unroll
        for (int q = 0; q < N; ++q) {
          ss = fmaf(p[r][q], p[r][q], ss);
          dot = fmaf(wq[q], p[r][q], dot);
        }
      }
      ss = warp_sum(ss);
      dot = warp_sum(dot);
      if (lane == 0) {
        red[par][r][warp][0] = ss;
        red[par][r][warp][1] = dot;
      }
    }
    __syncthreads();
#pragma unroll
    for (int r = 0; r < kRows; ++r) {
      if (!live[r]) continue;
      const int64_t row = base + r * rpb + slot;
      float tss = 0.f, tdot = 0.f;
      for (int w = 0; w < wpr; ++w) {
        tss += red[par][r][slot * wpr + w][0];
        tdot += red[par][r][slot * wpr + w][1];
      }
      const float s = tdot * rsqrtf(tss * inv_d + a.eps);
      const float lse = a.lse[row];
      const float M = fmaxf(lse, s);
      const float ea = __expf(lse - M), eb = __expf(s - M);
      const float inv = 1.0f / (ea + eb);
      const float ca = ea * inv, cb = eb * inv;
      float res[N];
#pragma unroll
      for (int q = 0; q < N; ++q) res[q] = fmaf(ca, o[r][q], cb * p[r][q]);
      Chunk<T>::store(static_cast<T*>(a.out) + row * d + k, res);
    }
  }
}

// ---------------------------------------------------------- general merge --

template <typename T>
__global__ void __launch_bounds__(kBlock) merge_generic_kernel(MergeArgs a) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int d = a.d;
  const float inv_d = 1.0f / static_cast<float>(d);
  for (int64_t row = static_cast<int64_t>(blockIdx.x) * kWarps + warp; row < a.T;
       row += static_cast<int64_t>(gridDim.x) * kWarps) {
    float ss = 0.f, dot = 0.f;
    for (int k = lane; k < d; k += 32) {
      const int64_t off = row * d + k;
      float p;
      if (a.f) {
        const float f = to_f32(static_cast<const T*>(a.f)[off]);
        p = a.p_empty ? f : a.P[off] + f;
        a.P[off] = p;
      } else {
        p = a.P[off];
      }
      ss = fmaf(p, p, ss);
      dot = fmaf(a.w[k] * a.gamma[k], p, dot);
    }
    ss = warp_sum(ss);
    dot = warp_sum(dot);
    const float s = dot * rsqrtf(ss * inv_d + a.eps);
    const float lse = a.lse[row];
    const float M = fmaxf(lse, s);
    const float ea = __expf(lse - M), eb = __expf(s - M);
    const float inv = 1.0f / (ea + eb);
    for (int k = lane; k < d; k += 32) {
      const int64_t off = row * d + k;
      const float o = to_f32(static_cast<const T*>(a.O)[off]);
      static_cast<T*>(a.out)[off] = from_f32<T>(fmaf(ea * inv, o, eb * inv * a.P[off]));
    }
  }
}

// ------------------------------------------------------- accumulate/freeze --

template <typename T>
__global__ void __launch_bounds__(kBlock) accum_fast_kernel(AccumArgs a, int64_t nchunks) {
  constexpr int N = Chunk<T>::N;
  pdl_trigger();
  pdl_wait();
  for (int64_t c = static_cast<int64_t>(blockIdx.x) * kBlock + threadIdx.x; c < nchunks;
       c += static_cast<int64_t>(gridDim.x) * kBlock) {
    const int64_t off = c * N;
    float f[N], p[N];
    Chunk<T>::load(static_cast<const T*>(a.f) + off, f);
    if (a.p_empty) {
#pragma unroll
      for (int q = 0; q < N; ++q) p[q] = f[q];
    } else {
      load_f32<N>(a.P + off, p);
#pragma unroll
      for (int q = 0; q < N; ++q) p[q] += f[q];
    }
    if (a.summary)
      Chunk<T>::store(static_cast<T*>(a.summary) + off, p);
    else
      store_f32<N>(a.P + off, p);
  }
}

template <typename T>
__global__ void __launch_bounds__(kBlock) accum_generic_kernel(AccumArgs a, int64_t n) {
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * kBlock + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * kBlock) {
    const float f = to_f32(static_cast<const T*>(a.f)[i]);
    const float p = a.p_empty ? f : a.P[i] + f;
    if (a.summary)
      static_cast<T*>(a.summary)[i] = from_f32<T>(p);
    else
      a.P[i] = p;
  }
}

int merge_wpr(int d, int bf16) {
  const int n = bf16 ? 8 : 4;
  const int warps = (d / n + 31) / 32;
  int wpr = 1;
  while (wpr < warps) wpr <<= 1;
  return wpr;
}

// Enough blocks for the work, at most one resident wave of `kernel`.
unsigned grid_for(int64_t work_items, int per_block, const void* kernel) {
  int64_t blocks = (work_items + per_block - 1) / per_block;
  const int64_t cap = static_cast<int64_t>(sm_count()) * blocks_per_sm(kernel, kBlock, 0);
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  return static_cast<unsigned>(blocks);
}

}  // namespace

bool merge_fast_ok(const MergeArgs& a) {
  const int n = a.bf16 ? 8 : 4;
  if (a.d % n != 0 || merge_wpr(a.d, a.bf16) > kWarps) return false;
  return aligned16(a.O) && aligned16(a.P) && aligned16(a.out) && (a.f == nullptr || aligned16(a.f));
}

bool accum_fast_ok(const AccumArgs& a) {
  const int n = a.bf16 ? 8 : 4;
  if (a.d % n != 0) return false;
  return aligned16(a.P) && aligned16(a.f) && (a.summary == nullptr || aligned16(a.summary));
}

cudaError_t launch_merge(const MergeArgs& a, cudaStream_t s, bool fast) {
  if (fast) {
    const int wpr = merge_wpr(a.d, a.bf16);
    const int rows_per_block = kWarps / wpr * kRows;
    if (a.bf16) {
      auto k = merge_fast_kernel<bf16>;
      return launch_pdl(k, grid_for(a.T, rows_per_block, reinterpret_cast<const void*>(k)), kBlock, 0, s, a, wpr);
    }
    auto k = merge_fast_kernel<float>;
    return launch_pdl(k, grid_for(a.T, rows_per_block, reinterpret_cast<const void*>(k)), kBlock, 0, s, a, wpr);
  }
  if (a.bf16) {
    auto k = merge_generic_kernel<bf16>;
    k<<<grid_for(a.T, kWarps, reinterpret_cast<const void*>(k)), kBlock, 0, s>>>(a);
  } else {
    auto k = merge_generic_kernel<float>;
    k<<<grid_for(a.T, kWarps, reinterpret_cast<const void*>(k)), kBlock, 0, s>>>(a);
  }
  return cudaGetLastError();
}

cudaError_t launch_accum(const AccumArgs& a, cudaStream_t s, bool fast) {
  const int64_t total = a.T * a.d;
  if (fast) {
    const int64_t nchunks = total / (a.bf16 ? 8 : 4);
    if (a.bf16) {
      auto k = accum_fast_kernel<bf16>;
      return launch_pdl(k, grid_for(nchunks, kBlock, reinterpret_cast<const void*>(k)), kBlock, 0, s, a, nchunks);
    }
    auto k = accum_fast_kernel<float>;
    return launch_pdl(k, grid_for(nchunks, kBlock, reinterpret_cast<const void*>(k)), kBlock, 0, s, a, nchunks);
  }
  if (a.bf16) {
    auto k = accum_generic_kernel<bf16>;
    k<<<grid_for(total, kBlock, reinterpret_cast<const void*>(k)), kBlock, 0, s>>>(a, total);
  } else {
    auto k = accum_generic_kernel<float>;
    k<<<grid_for(total, kBlock, reinterpret_cast<const void*>(k)), kBlock, 0, s>>>(a, total);
  }
  return cudaGetLastError();
}

}  // namespace attnres
