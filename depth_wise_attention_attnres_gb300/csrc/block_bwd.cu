// Elementwise kernels of the Block pass backward (attnres_block_bwd in api.cu
// drives them around the per-read backward of full_bwd.cu).
//
// The Block pass reads, for sublayer k = n * S + j, the sources {embedding,
// b_1 .. b_n, P_k if j >= 1} (DepthBench reading notes section 2.5; LLMRes
// blog, "Block Attention Residuals"): b_m is the plain sum of block (m-1)'s
// outputs and P_k the sum of the earlier outputs of block n. By the chain rule
// the gradient of b_m reaches every member of block m-1 unchanged, and that of
// P_k every output of block n before k. The backward runs the reads in
// reverse order over fp32 copies of the sources; these kernels widen the
// sources, rebuild the running sums as the forward formed them (the same fp32
// additions in the same order), and route the summaries' and running sums'
// gradients to the outputs.
#include <initializer_list>

#include "common.cuh"
#include "internal.h"

namespace attnres {
namespace {

constexpr int kEwThreads = 256;

inline unsigned ew_grid(int64_t n4) {
  int64_t g = (n4 + kEwThreads - 1) / kEwThreads;
  const int64_t cap = static_cast<int64_t>(sm_count()) * 8;
  if (g > cap) g = cap;
  return static_cast<unsigned>(g > 0 ? g : 1);
}

// Grid-stride loop over groups of 4 elements (n a multiple of 4, 16-byte
// aligned rows), else over single elements.
#define EW_LOOP(i, n)                                                                       \
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < (n); \
       i += static_cast<int64_t>(gridDim.x) * blockDim.x)

template <typename T>
__global__ void widen_rows_kernel(const T* src, int64_t src_stride, float* dst, int R, int64_t E, bool vec) {
  for (int r = 0; r < R; ++r) {
    const T* s = src + r * src_stride;
    float* o = dst + r * E;
    if (vec) {
      EW_LOOP(i, E / 4) {
        float x[4];
        ldg4(s + i * 4, x);
        st4(o + i * 4, x);
      }
    } else {
      EW_LOOP(i, E) o[i] = to_f32(s[i]);
    }
  }
}

// dst = prev + f (prev null: dst = f).
template <typename T>
__global__ void psum_kernel(float* dst, const float* prev, const T* f, int64_t E, bool vec) {
  if (vec) {
    EW_LOOP(i, E / 4) {
      float x[4];
      ldg4(f + i * 4, x);
      if (prev) {
        const float4 p = reinterpret_cast<const float4*>(prev)[i];
        x[0] = p.x + x[0]; x[1] = p.y + x[1]; x[2] = p.z + x[2]; x[3] = p.w + x[3];
      }
      st4(dst + i * 4, x);
    }
  } else {
    EW_LOOP(i, E) dst[i] = prev ? prev[i] + to_f32(f[i]) : to_f32(f[i]);
  }
}

// G += ds; dF_prev += G; ds = 0.
__global__ void gupdate_kernel(float* G, float* ds, float* dfp, int64_t E, bool vec) {
  if (vec) {
    EW_LOOP(i, E / 4) {
      float4 g = reinterpret_cast<float4*>(G)[i];
      const float4 s = reinterpret_cast<const float4*>(ds)[i];
      float4 f = reinterpret_cast<float4*>(dfp)[i];
      g.x += s.x; g.y += s.y; g.z += s.z; g.w += s.w;
      f.x += g.x; f.y += g.y; f.z += g.z; f.w += g.w;
      reinterpret_cast<float4*>(G)[i] = g;
      reinterpret_cast<float4*>(dfp)[i] = f;
      reinterpret_cast<float4*>(ds)[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
  } else {
    EW_LOOP(i, E) {
      G[i] += ds[i];
      dfp[i] += G[i];
      ds[i] = 0.f;
    }
  }
}

// dst[q] += g for q < R rows dst_stride apart.
__global__ void spread_kernel(float* dst, int64_t dst_stride, int R, const float* g, int64_t E, bool vec) {
  if (vec) {
    EW_LOOP(i, E / 4) {
      const float4 v = reinterpret_cast<const float4*>(g)[i];
      for (int q = 0; q < R; ++q) {
        float4* o = reinterpret_cast<float4*>(dst + q * dst_stride) + i;
        float4 x = *o;
        x.x += v.x; x.y += v.y; x.z += v.z; x.w += v.w;
        *o = x;
      }
    }
  } else {
    EW_LOOP(i, E) {
      const float v = g[i];
      for (int q = 0; q < R; ++q) dst[q * dst_stride + i] += v;
    }
  }
}

#undef EW_LOOP

inline bool vec_ok(int64_t E, std::initializer_list<const void*> ptrs, std::initializer_list<int64_t> strides) {
  if (E % 4 != 0) return false;
  for (const void* p : ptrs)
    if (p && !aligned16(p)) return false;
  for (int64_t s : strides)
    if (s % 4 != 0) return false;
  return true;
}

}  // namespace

cudaError_t launch_widen_rows(const void* src, int64_t src_stride, int is_bf16, float* dst, int R, int64_t E,
                              cudaStream_t s) {
  const bool vec = vec_ok(E, {src, dst}, {src_stride});
  const unsigned g = ew_grid(vec ? E / 4 : E);
  if (is_bf16)
    widen_rows_kernel<bf16><<<g, kEwThreads, 0, s>>>(static_cast<const bf16*>(src), src_stride, dst, R, E, vec);
  else
    widen_rows_kernel<float><<<g, kEwThreads, 0, s>>>(static_cast<const float*>(src), src_stride, dst, R, E, vec);
  return cudaGetLastError();
}

cudaError_t launch_psum(float* dst, const float* prev, const void* f, int is_bf16, int64_t E, cudaStream_t s) {
  const bool vec = vec_ok(E, {dst, prev, f}, {});
  const unsigned g = ew_grid(vec ? E / 4 : E);
  if (is_bf16)
    psum_kernel<bf16><<<g, kEwThreads, 0, s>>>(dst, prev, static_cast<const bf16*>(f), E, vec);
  else
    psum_kernel<float><<<g, kEwThreads, 0, s>>>(dst, prev, static_cast<const float*>(f), E, vec);
  return cudaGetLastError();
}

cudaError_t launch_gupdate(float* G, float* ds, float* dfp, int64_t E, cudaStream_t s) {
  const bool vec = vec_ok(E, {G, ds, dfp}, {});
  gupdate_kernel<<<ew_grid(vec ? E / 4 : E), kEwThreads, 0, s>>>(G, ds, dfp, E, vec);
  return cudaGetLastError();
}

cudaError_t launch_spread(float* dst, int64_t dst_stride, int R, const float* g, int64_t E, cudaStream_t s) {
  const bool vec = vec_ok(E, {dst, g}, {dst_stride});
  spread_kernel<<<ew_grid(vec ? E / 4 : E), kEwThreads, 0, s>>>(dst, dst_stride, R, g, E, vec);
  return cudaGetLastError();
}

}  // namespace attnres
