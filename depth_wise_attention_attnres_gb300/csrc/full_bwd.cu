// Backward of one AttnRes read: the gradients with respect to its sources,
// its query w and its key-norm gain gamma, given dz = dL/dz of its result.
//
// The read (DepthBench reading notes section 2.3): e_i = r_i (u . v_i) with
// u = w * gamma and r_i = 1 / sqrt(mean_k v_ik^2 + eps), a = softmax_i(e),
// z = sum_i a_i v_i. By the chain rule, per token:
//   dL/da_i = dz . v_i,   gbar = sum_j a_j dL/da_j,   dL/de_i = a_i (dL/da_i - gbar)
//   dL/dv_i = a_i dz + dL/de_i r_i u - dL/de_i e_i r_i^2 / d v_i
//   dL/du  += dL/de_i r_i v_i   (summed over tokens; dw = du * gamma, dgamma = du * w)
// dV, dw and dgamma are accumulated (+=) in fp32: a model's backward adds the
// contributions of every later read to a source's gradient.
//
// full_bwd_bulk_kernel: the Full-read pipeline run twice per tile of 8 token
// rows (one consumer warp per row). A producer warp streams every (tile,
// source) block with one bulk copy, first for pass A and again for pass B (the
// second pass takes the sources in reverse order, so its first blocks are
// the ones still in L2). Pass A forms Sigma v^2, u . v and dz . v per source with
// packed FMAs and warp sums and keeps e_i, dz . v_i and r_i in shared memory
// while an online softmax gathers the max, the mass and sum_i a_i dL/da_i.
// The per-source coefficients then turn dv_i into A_i dz + B_i u + C_i v_i
// (A = a_i, B = dL/de_i r_i, C = -dL/de_i e_i r_i^2 / d), which pass B
// applies, adding into dV with 16-byte atomic adds (the L2 does the read-
// modify-write) and into the per-lane du registers. du is reduced per CTA in
// shared memory and added to dw and dgamma once per feature.
#include <math.h>

#include "common.cuh"
#include "internal.h"

namespace attnres {
namespace {

__device__ unsigned int g_bwd_timeout = 0;

constexpr int kBNW = 8;                       // consumer warps = rows per tile
constexpr int kBThreads = (kBNW + 1) * kWarp;  // + producer warp
constexpr int kBBar = 128;
constexpr int kBMaxStages = 8;
constexpr int kBSmemPerSM = 224 * 1024;

// One CTA per SM: with two, the tiles of all CTAs together (8 rows of every
// source each) outgrew the L2 sooner, and more of pass B's reads went to DRAM
// (measured: 64-read 8192 x 896 pass backward 26.97 ms with two CTAs per SM,
// 26.72 ms with one; 4-row tiles were slower at two or four CTAs per SM).
template <int CH>
struct BwdTraits {
  static constexpr int kMinBlocks = 1;
};

struct BwdGeom {
  int nstage;
  int wq_off, du_off, g_off, sc_off, stage_off, total;
};

inline int round_up_b(int x, int m) { return (x + m - 1) / m * m; }

template <typename Tin, int CH>
BwdGeom bwd_geom(int n) {
  constexpr int D = CH * 128;
  BwdGeom g{};
  g.wq_off = kBBar;                      // w * gamma [D]
  g.du_off = g.wq_off + D * 4;           // du partial sums of the CTA [D]
  g.g_off = g.du_off + D * 4;            // dz rows in fp32 [kBNW][D]
  g.sc_off = g.g_off + kBNW * D * 4;     // per (row, source): e, dz.v, r, then A, B, C [kBNW][n][3]
  g.stage_off = round_up_b(g.sc_off + kBNW * n * 3 * 4, 128);
  const int stage_bytes = kBNW * D * static_cast<int>(sizeof(Tin));
  int ns = (kBSmemPerSM / BwdTraits<CH>::kMinBlocks - 1024 - g.stage_off) / stage_bytes;
  g.nstage = ns < 2 ? 2 : (ns > kBMaxStages ? kBMaxStages : ns);
  g.total = g.stage_off + g.nstage * stage_bytes;
  return g;
}

// L2 eviction priorities for the two passes over a tile's sources: pass A
// marks the rows it brings in to be kept (pass B reads them again soon), pass
// B and the dV reductions mark theirs to go first. Without them the dV
// read-modify-write stream pushed part of the sources out of the L2 between
// the passes, and pass B re-read them from DRAM.
__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// 1-D bulk copy global -> shared with an L2 eviction priority.
__device__ __forceinline__ void bulk_g2s_hint(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar,
                                              uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
          dst),
      "l"(src), "r"(bytes), "r"(bar), "l"(policy)
      : "memory");
}

__device__ __forceinline__ void red_add4(float* p, const float (&x)[4], uint64_t policy) {
  asm volatile("red.global.add.L2::cache_hint.v4.f32 [%0], {%1, %2, %3, %4}, %5;" ::"l"(p), "f"(x[0]), "f"(x[1]),
               "f"(x[2]), "f"(x[3]), "l"(policy)
               : "memory");
}

template <typename T>
__device__ __forceinline__ void ldg4_any(const T* p, float (&x)[4]) {
  if constexpr (sizeof(T) == 2) {
    const uint2 v = *reinterpret_cast<const uint2*>(p);
    x[0] = bf16_lo(v.x); x[1] = bf16_hi(v.x); x[2] = bf16_lo(v.y); x[3] = bf16_hi(v.y);
  } else {
    const float4 v = *reinterpret_cast<const float4*>(p);
    x[0] = v.x; x[1] = v.y; x[2] = v.z; x[3] = v.w;
  }
}

template <typename Tin, int CH>
__global__ void __launch_bounds__(kBThreads, BwdTraits<CH>::kMinBlocks)
    full_bwd_bulk_kernel(BwdArgs a, BwdGeom g) {
  constexpr int D = CH * 128;
  constexpr int NE = CH * 4;
  extern __shared__ __align__(128) unsigned char smem[];
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem);
  uint64_t* empty_bar = full_bar + kBMaxStages;
  float* wq = reinterpret_cast<float*>(smem + g.wq_off);
  float* duacc = reinterpret_cast<float*>(smem + g.du_off);
  float* gsm = reinterpret_cast<float*>(smem + g.g_off);
  float* scs = reinterpret_cast<float*>(smem + g.sc_off);
  Tin* stages = reinterpret_cast<Tin*>(smem + g.stage_off);
  constexpr int kStageElems = kBNW * D;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n = a.n_src;
  const int nstage = g.nstage;
  const int64_t T = a.T;
  const int64_t r0 = static_cast<int64_t>(blockIdx.x) * T / gridDim.x;
  const int64_t r1 = static_cast<int64_t>(blockIdx.x + 1) * T / gridDim.x;
  const int R = static_cast<int>(r1 - r0);
  const int ntiles = (R + kBNW - 1) / kBNW;
  const int64_t total = static_cast<int64_t>(ntiles) * 2 * n;

  pdl_trigger();
  if (threadIdx.x == 0) {
    for (int s = 0; s < nstage; ++s) {
      mbar_init(smem_u32(&full_bar[s]), 1);
      mbar_init(smem_u32(&empty_bar[s]), kBNW);
    }
    mbar_fence_init();
  }
  __syncthreads();
  pdl_wait();  // everything below may read what the previous kernel wrote

  if (warp == kBNW) {
    // ------------------------------------------------------------ producer
    if (lane != 0) return;
    const char* V = static_cast<const char*>(a.V);
    const uint64_t keep = policy_evict_last(), drop = policy_evict_first();
    int stage = 0;
    uint32_t phase = 0;
    int64_t issued = 0;
    bool ok = true;
    for (int64_t it = 0; it < total; ++it) {
      if (!mbar_wait(smem_u32(&empty_bar[stage]), phase ^ 1u)) {
        ok = false;
        break;
      }
      const int tile = static_cast<int>(it / (2 * n));
      // Pass A in source order, pass B in reverse (its first blocks are the
      // ones pass A brought in last, the likeliest still in L2).
      const int j = static_cast<int>(it - static_cast<int64_t>(tile) * 2 * n);
      const int src = j < n ? j : 2 * n - 1 - j;
      const int64_t row0 = r0 + static_cast<int64_t>(tile) * R / ntiles;
      const int rows = static_cast<int>(r0 + static_cast<int64_t>(tile + 1) * R / ntiles - row0);
      const uint32_t bytes = static_cast<uint32_t>(rows) * D * sizeof(Tin);
      const uint32_t fb = smem_u32(&full_bar[stage]);
      mbar_arrive_expect_tx(fb, bytes);
      bulk_g2s_hint(smem_u32(stages + static_cast<size_t>(stage) * kStageElems),
                    V + (static_cast<int64_t>(src) * a.src_stride + row0 * D) * sizeof(Tin), bytes, fb,
                    j < n ? keep : drop);
      ++issued;
      if (++stage == nstage) {
        stage = 0;
        phase ^= 1u;
      }
    }
    if (!ok) {
      atomicOr(&g_bwd_timeout, 1u);
      // Let the copies still in flight land before this CTA's memory goes.
      for (int64_t it = issued > nstage ? issued - nstage : 0; it < issued; ++it)
        (void)mbar_wait(smem_u32(&full_bar[it % nstage]), static_cast<uint32_t>((it / nstage) & 1));
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  for (int i = threadIdx.x; i < D; i += kBNW * kWarp) {
    wq[i] = a.w[i] * a.gamma[i];
    duacc[i] = 0.f;
  }
  named_sync(1, kBNW * kWarp);
  const float inv_d = 1.0f / static_cast<float>(D);
  const uint64_t dv_policy = policy_evict_first();
  float* grow = gsm + warp * D;
  float* sc = scs + warp * n * 3;
  float2 du[NE / 2];
#pragma unroll
  for (int e = 0; e < NE / 2; ++e) du[e] = make_float2(0.f, 0.f);

  int stage = 0;
  uint32_t phase = 0;
  bool ok = true;
  for (int tile = 0; tile < ntiles && ok; ++tile) {
    const int64_t row0 = r0 + static_cast<int64_t>(tile) * R / ntiles;
    const int64_t row = row0 + warp;
    const bool valid = row < r0 + static_cast<int64_t>(tile + 1) * R / ntiles;
    if (valid) {
#pragma unroll
      for (int c = 0; c < CH; ++c) {
        const int k = (c * kWarp + lane) * 4;
        float x[4];
        if (a.dz_bf16)
          ldg4_any(static_cast<const bf16*>(a.dz) + row * D + k, x);
        else
          ldg4_any(static_cast<const float*>(a.dz) + row * D + k, x);
        st4(grow + k, x);
      }
    }
    __syncwarp();

    // Pass A: scores, dz . v, and the online softmax statistics.
    float m = -INFINITY, z = 0.f, sa = 0.f;
    for (int src = 0; src < n && ok; ++src) {
      if (!mbar_wait(smem_u32(&full_bar[stage]), phase)) {
        ok = false;
        break;
      }
      if (valid) {
        const Tin* rowp = stages + static_cast<size_t>(stage) * kStageElems + warp * D;
        float2 ss2 = make_float2(0.f, 0.f), ud2 = ss2, gd2 = ss2;
#pragma unroll
        for (int c = 0; c < CH; ++c) {
          const int k = (c * kWarp + lane) * 4;
          float x[4], gz[4];
          lds4(rowp + k, x);
          lds4(grow + k, gz);
          const float4 w4 = *reinterpret_cast<const float4*>(wq + k);
          const float2 xa = make_float2(x[0], x[1]), xb = make_float2(x[2], x[3]);
          ss2 = ffma2(xa, xa, ss2);
          ss2 = ffma2(xb, xb, ss2);
          ud2 = ffma2(make_float2(w4.x, w4.y), xa, ud2);
          ud2 = ffma2(make_float2(w4.z, w4.w), xb, ud2);
          gd2 = ffma2(make_float2(gz[0], gz[1]), xa, gd2);
          gd2 = ffma2(make_float2(gz[2], gz[3]), xb, gd2);
        }
        const float ss = warp_sum(ss2.x + ss2.y);
        const float ud = warp_sum(ud2.x + ud2.y);
        const float gd = warp_sum(gd2.x + gd2.y);
        const float r = rsqrtf(ss * inv_d + a.eps);
        const float s = ud * r;
        if (lane == 0) {
          sc[src * 3 + 0] = s;
          sc[src * 3 + 1] = gd;
          sc[src * 3 + 2] = r;
        }
        if (s > m) {  // warp-uniform
          const float cfac = __expf(m - s);
          z *= cfac;
          sa *= cfac;
          m = s;
        }
        const float p = __expf(s - m);
        z += p;
        sa = fmaf(p, gd, sa);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&empty_bar[stage]));
      if (++stage == nstage) {
        stage = 0;
        phase ^= 1u;
      }
    }
    if (!ok) break;

    // Per-source coefficients of dv_i = A dz + B u + C v_i.
    if (valid) {
      const float invz = 1.0f / z;
      const float gbar = sa * invz;
      __syncwarp();
      for (int src = lane; src < n; src += kWarp) {
        const float s = sc[src * 3 + 0], gd = sc[src * 3 + 1], r = sc[src * 3 + 2];
        const float al = __expf(s - m) * invz;
        const float de = al * (gd - gbar);
        sc[src * 3 + 0] = al;
        sc[src * 3 + 1] = de * r;
        sc[src * 3 + 2] = -de * s * r * r * inv_d;
      }
      __syncwarp();
    }

    // Pass B (sources in reverse): dv_i into dV, du into registers.
    for (int src = n - 1; src >= 0 && ok; --src) {
      if (!mbar_wait(smem_u32(&full_bar[stage]), phase)) {
        ok = false;
        break;
      }
      if (valid) {
        const Tin* rowp = stages + static_cast<size_t>(stage) * kStageElems + warp * D;
        const float A = sc[src * 3 + 0], B = sc[src * 3 + 1], C = sc[src * 3 + 2];
        float* dvrow = a.dV + src * a.dv_stride + row * D;
        const float2 A2 = make_float2(A, A), B2 = make_float2(B, B), C2 = make_float2(C, C);
#pragma unroll
        for (int c = 0; c < CH; ++c) {
          const int k = (c * kWarp + lane) * 4;
          float x[4], gz[4];
          lds4(rowp + k, x);
          lds4(grow + k, gz);
          const float4 w4 = *reinterpret_cast<const float4*>(wq + k);
          const float2 xa = make_float2(x[0], x[1]), xb = make_float2(x[2], x[3]);
          float2 va = fmul2(A2, make_float2(gz[0], gz[1]));
          float2 vb = fmul2(A2, make_float2(gz[2], gz[3]));
          va = ffma2(B2, make_float2(w4.x, w4.y), va);
          vb = ffma2(B2, make_float2(w4.z, w4.w), vb);
          va = ffma2(C2, xa, va);
          vb = ffma2(C2, xb, vb);
          const float dv[4] = {va.x, va.y, vb.x, vb.y};
          red_add4(dvrow + k, dv, dv_policy);
          du[c * 2] = ffma2(B2, xa, du[c * 2]);
          du[c * 2 + 1] = ffma2(B2, xb, du[c * 2 + 1]);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&empty_bar[stage]));
      if (++stage == nstage) {
        stage = 0;
        phase ^= 1u;
      }
    }
  }

  // du of this CTA: warps meet in shared memory, then one add per feature.
#pragma unroll
  for (int c = 0; c < CH; ++c) {
    const int k = (c * kWarp + lane) * 4;
    atomicAdd(duacc + k, du[c * 2].x);
    atomicAdd(duacc + k + 1, du[c * 2].y);
    atomicAdd(duacc + k + 2, du[c * 2 + 1].x);
    atomicAdd(duacc + k + 3, du[c * 2 + 1].y);
  }
  named_sync(1, kBNW * kWarp);
  for (int k = threadIdx.x; k < D; k += kBNW * kWarp) {
    if (a.dw) atomicAdd(a.dw + k, duacc[k] * a.gamma[k]);
    if (a.dgamma) atomicAdd(a.dgamma + k, duacc[k] * a.w[k]);
  }
  if (!ok) atomicOr(&g_bwd_timeout, 1u);
}

// General shapes: one warp per token row, two passes over the sources read
// from global memory (the second recomputes the scalars), du in shared memory.
template <typename T, typename TZ>
__global__ void __launch_bounds__(256) full_bwd_generic_kernel(BwdArgs a) {
  extern __shared__ float dus[];  // [d]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int d = a.d, n = a.n_src;
  pdl_trigger();
  for (int k = threadIdx.x; k < d; k += blockDim.x) dus[k] = 0.f;
  __syncthreads();
  pdl_wait();
  const float inv_d = 1.0f / static_cast<float>(d);
  const T* V = static_cast<const T*>(a.V);
  const TZ* dz = static_cast<const TZ*>(a.dz);
  for (int64_t row = static_cast<int64_t>(blockIdx.x) * 8 + warp; row < a.T;
       row += static_cast<int64_t>(gridDim.x) * 8) {
    auto scalars = [&](int i, float& s, float& gd, float& r) {
      const T* v = V + i * a.src_stride + row * d;
      float ss = 0.f, ud = 0.f, g = 0.f;
      for (int k = lane; k < d; k += kWarp) {
        const float x = to_f32(v[k]);
        ss = fmaf(x, x, ss);
        ud = fmaf(a.w[k] * a.gamma[k], x, ud);
        g = fmaf(to_f32(dz[row * d + k]), x, g);
      }
      r = rsqrtf(warp_sum(ss) * inv_d + a.eps);
      s = warp_sum(ud) * r;
      gd = warp_sum(g);
    };
    float m = -INFINITY, z = 0.f, sa = 0.f;
    for (int i = 0; i < n; ++i) {
      float s, gd, r;
      scalars(i, s, gd, r);
      if (s > m) {
        const float cfac = __expf(m - s);
        z *= cfac;
        sa *= cfac;
        m = s;
      }
      const float p = __expf(s - m);
      z += p;
      sa = fmaf(p, gd, sa);
    }
    const float invz = 1.0f / z, gbar = sa * invz;
    for (int i = 0; i < n; ++i) {
      float s, gd, r;
      scalars(i, s, gd, r);
      const float al = __expf(s - m) * invz;
      const float de = al * (gd - gbar);
      const float B = de * r, C = -de * s * r * r * inv_d;
      const T* v = V + i * a.src_stride + row * d;
      float* dvrow = a.dV + i * a.dv_stride + row * d;
      for (int k = lane; k < d; k += kWarp) {
        const float x = to_f32(v[k]);
        atomicAdd(dvrow + k, al * to_f32(dz[row * d + k]) + B * a.w[k] * a.gamma[k] + C * x);
        atomicAdd(dus + k, B * x);
      }
    }
  }
  __syncthreads();
  for (int k = threadIdx.x; k < d; k += blockDim.x) {
    if (a.dw) atomicAdd(a.dw + k, dus[k] * a.gamma[k]);
    if (a.dgamma) atomicAdd(a.dgamma + k, dus[k] * a.w[k]);
  }
}

template <typename Tin, int CH>
cudaError_t launch_bwd_ch(const BwdArgs& a, cudaStream_t s) {
  const BwdGeom g = bwd_geom<Tin, CH>(a.n_src);
  auto k = full_bwd_bulk_kernel<Tin, CH>;
  cudaError_t e = allow_dynamic_smem(reinterpret_cast<const void*>(k), g.total);
  if (e != cudaSuccess) return e;
  const int per_sm = blocks_per_sm(reinterpret_cast<const void*>(k), kBThreads, g.total);
  const int64_t tiles = (a.T + kBNW - 1) / kBNW;
  int64_t grid = static_cast<int64_t>(sm_count()) * (per_sm > 0 ? per_sm : 1);
  if (grid > tiles) grid = tiles;
  return launch_pdl(k, static_cast<unsigned>(grid), kBThreads, g.total, s, a, g);
}

template <typename Tin>
cudaError_t launch_bwd_dtype(const BwdArgs& a, cudaStream_t s) {
  switch (a.d / 128) {
    case 1: return launch_bwd_ch<Tin, 1>(a, s);
    case 2: return launch_bwd_ch<Tin, 2>(a, s);
    case 4: return launch_bwd_ch<Tin, 4>(a, s);
    case 5: return launch_bwd_ch<Tin, 5>(a, s);
    case 6: return launch_bwd_ch<Tin, 6>(a, s);
    case 7: return launch_bwd_ch<Tin, 7>(a, s);
    case 8: return launch_bwd_ch<Tin, 8>(a, s);
    case 16: return launch_bwd_ch<Tin, 16>(a, s);
    default: return cudaErrorInvalidValue;
  }
}

template <typename T, typename TZ>
cudaError_t launch_bwd_generic_t(const BwdArgs& a, cudaStream_t s) {
  const int smem = a.d * 4;
  auto k = full_bwd_generic_kernel<T, TZ>;
  cudaError_t e = allow_dynamic_smem(reinterpret_cast<const void*>(k), smem);
  if (e != cudaSuccess) return e;
  int64_t blocks = (a.T + 7) / 8;
  const int64_t cap = static_cast<int64_t>(sm_count()) * 8;
  if (blocks > cap) blocks = cap;
  return launch_pdl(k, static_cast<unsigned>(blocks), 256, smem, s, a);
}

}  // namespace

bool full_bwd_fast_ok(const BwdArgs& a) {
  const int ch = a.d / 128;
  const bool ch_ok = a.d % 128 == 0 && (ch == 1 || ch == 2 || (ch >= 4 && ch <= 8) || ch == 16);
  const int es = a.v_bf16 ? 2 : 4;
  if (!ch_ok || a.n_src > kMaxBwdFastSources) return false;
  return aligned16(a.V) && aligned16(a.dz) && aligned16(a.dV) && aligned16(a.w) && aligned16(a.gamma) &&
         (a.src_stride * es) % 16 == 0 && (a.dv_stride * 4) % 16 == 0;
}

cudaError_t launch_full_bwd(const BwdArgs& a, cudaStream_t s, bool fast) {
  if (fast) return a.v_bf16 ? launch_bwd_dtype<bf16>(a, s) : launch_bwd_dtype<float>(a, s);
  if (a.d > kMaxBwdGenericD) return cudaErrorInvalidValue;
  if (a.v_bf16)
    return a.dz_bf16 ? launch_bwd_generic_t<bf16, bf16>(a, s) : launch_bwd_generic_t<bf16, float>(a, s);
  return a.dz_bf16 ? launch_bwd_generic_t<float, bf16>(a, s) : launch_bwd_generic_t<float, float>(a, s);
}

cudaError_t take_timeout_bwd(unsigned int* flag) {
  unsigned int zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(flag, g_bwd_timeout, sizeof(unsigned int));
  if (e != cudaSuccess) return e;
  return cudaMemcpyToSymbol(g_bwd_timeout, &zero, sizeof(unsigned int));
}

}  // namespace attnres
