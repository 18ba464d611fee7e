// Block AttnRes stage 1, fast kernel (sm_103a).
//
// Stage 1 of the two-stage computation (datacamp explainer, "two-stage
// computation"): the S pseudo-queries of one block read the n cross-block
// sources (embedding and completed block sums), and each source row is moved
// from HBM once for all S queries. For each query j and token row t it writes
// the normalised read O_j[t] = sum_i softmax_i(e_ij) v_i[t] and
// lse_j[t] = log sum_i exp(e_ij), e_ij = w_j^T RMSNorm_j(v_i[t]).
//
// A CTA processes tiles of TM token rows. For a tile, the n*TM source rows
// are brought into one of two shared-memory buffers by 1-D bulk copies, one
// per row into a pitch padded by 16 bytes (so rows start in different bank
// groups), while the other buffer is being computed on. Then, per tile:
//   A. scores: warp w owns a 1/8 slice of the features and lane p owns one
//      (source, row) pair; a lane runs over its slice with the S pseudo-
//      queries read as shared-memory broadcasts, so no cross-lane reduction
//      is needed; the 8 warp partials are summed through shared memory;
//   B. softmax over the n sources for every (row, query): weights and lse;
//   C. accumulation: threads own 4-feature chunks of a row and form all S
//      outputs from the staged rows (fp32 registers), written with 8/16-byte
//      stores.
// Sums of squares, dots and accumulations use packed fp32x2 FMAs.
#include <math.h>

#include "common.cuh"
#include "internal.h"

namespace attnres {
namespace {

__device__ unsigned int g_stage1_timeout = 0;

constexpr int kNW = 8;                       // consumer warps
constexpr int kConsumers = kNW * kWarp;      // 256
constexpr int kThreads = kConsumers + kWarp; // + producer warp
constexpr int kMaxPairs = 32;                // (source, row) pairs per tile
constexpr int kSmemLimit = 220 * 1024;
constexpr int kBarBytes = 128;

struct Stage1Geom {
  int TM;          // rows per tile
  int pitch;       // bytes between staged rows
  int buf_bytes;   // one buffer
  int w_off, red_off, alpha_off, buf_off, total;
};

__host__ __device__ inline int round_up(int x, int m) { return (x + m - 1) / m * m; }

inline Stage1Geom stage1_geom(int n, int d, int S, int es) {
  Stage1Geom g{};
  const int S4 = round_up(S, 4);
  g.pitch = d * es + 16;
  g.w_off = kBarBytes;
  g.red_off = g.w_off + S * d * 4;
  g.alpha_off = g.red_off + kNW * kMaxPairs * (S + 1) * 4;
  g.buf_off = round_up(g.alpha_off + kMaxPairs * S4 * 4, 128);
  const int avail = kSmemLimit - g.buf_off;
  int pmax = avail / 2 / g.pitch;
  if (pmax > kMaxPairs) pmax = kMaxPairs;
  g.TM = n > 0 ? pmax / n : 0;
  g.buf_bytes = g.TM * n * g.pitch;
  g.total = g.buf_off + 2 * g.buf_bytes;
  return g;
}

template <typename Tin, int S, int CPT>
__global__ void __launch_bounds__(kThreads, 1) stage1_kernel(MultiArgs a, Stage1Geom g) {
  constexpr int VEC = 16 / sizeof(Tin);      // elements per 16-byte load
  constexpr int S4 = (S + 3) / 4 * 4;
  extern __shared__ __align__(128) unsigned char smem[];
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem);
  uint64_t* empty_bar = full_bar + 2;
  float* wq = reinterpret_cast<float*>(smem + g.w_off);        // [S][d]
  float* red = reinterpret_cast<float*>(smem + g.red_off);     // [kNW][kMaxPairs][S+1]
  float* alpha = reinterpret_cast<float*>(smem + g.alpha_off); // [TM][n][S4]
  unsigned char* bufs = smem + g.buf_off;

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int n = a.n_src, d = a.d, TM = g.TM;
  const int P = TM * n;
  const int64_t T = a.T;
  const int64_t ntiles_total = (T + TM - 1) / TM;
  // Contiguous tile range per CTA.
  const int64_t t0 = static_cast<int64_t>(blockIdx.x) * ntiles_total / gridDim.x;
  const int64_t t1 = static_cast<int64_t>(blockIdx.x + 1) * ntiles_total / gridDim.x;

  pdl_trigger();
  if (tid == 0) {
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&full_bar[b]), 1);
      mbar_init(smem_u32(&empty_bar[b]), kNW);
    }
    *reinterpret_cast<int*>(full_bar + 4) = 0;  // consumer abort flag
    mbar_fence_init();
  }
  pdl_wait();  // global reads below may depend on the previous kernel
  // w * gamma for the S queries of the block.
  for (int idx = tid; idx < S * d / 4; idx += kThreads) {
    const float4 w4 = reinterpret_cast<const float4*>(a.W)[idx];
    const float4 g4 = reinterpret_cast<const float4*>(a.Gamma)[idx];
    reinterpret_cast<float4*>(wq)[idx] = make_float4(w4.x * g4.x, w4.y * g4.y, w4.z * g4.z, w4.w * g4.w);
  }
  __syncthreads();

  if (warp == kNW) {
    // ------------------------------------------------------------ producer
    if (lane != 0) return;
    const char* src = static_cast<const char*>(a.V);
    const uint32_t row_bytes = static_cast<uint32_t>(d) * sizeof(Tin);
    int b = 0;
    uint32_t phase = 0;
    int64_t issued = 0;
    bool ok = true;
    for (int64_t tile = t0; tile < t1; ++tile) {
      if (!mbar_wait(smem_u32(&empty_bar[b]), phase ^ 1u)) {
        ok = false;
        break;
      }
      const int64_t row0 = tile * TM;
      const int rows = static_cast<int>(min(static_cast<int64_t>(TM), T - row0));
      const uint32_t fb = smem_u32(&full_bar[b]);
      mbar_arrive_expect_tx(fb, row_bytes * rows * n);
      const uint32_t dst0 = smem_u32(bufs + b * g.buf_bytes);
      for (int i = 0; i < n; ++i)
        for (int r = 0; r < rows; ++r)
          bulk_g2s(dst0 + (i * TM + r) * g.pitch,
                   src + (i * a.src_stride + (row0 + r) * d) * static_cast<int64_t>(sizeof(Tin)),
                   row_bytes, fb);
      ++issued;
      if (++b == 2) {
        b = 0;
        phase ^= 1u;
      }
    }
    if (!ok) {
      atomicOr(&g_stage1_timeout, 1u);
      for (int64_t it = issued > 2 ? issued - 2 : 0; it < issued; ++it)
        (void)mbar_wait(smem_u32(&full_bar[it % 2]), static_cast<uint32_t>((it / 2) & 1));
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const float inv_d = 1.0f / static_cast<float>(d);
  const int KW = d / kNW;  // features per warp in the score pass
  int b = 0;
  uint32_t phase = 0;
  bool ok = true;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(full_bar + 4);
  for (int64_t tile = t0; tile < t1; ++tile) {
    // The consumers meet at named barriers below, so giving up a wait has to
    // be a joint decision: whoever times out raises a shared flag, and every
    // consumer reads it after the next barrier.
    if (!mbar_wait(smem_u32(&full_bar[b]), phase)) *abort_flag = 1;
    named_sync(1, kConsumers);
    if (*abort_flag) {
      ok = false;
      break;
    }
    const unsigned char* buf = bufs + b * g.buf_bytes;
    const int64_t row0 = tile * TM;
    const int rows = static_cast<int>(min(static_cast<int64_t>(TM), T - row0));

    // A. partial sums of squares and dots over this warp's feature slice.
    if (lane < P) {
      const Tin* rowp = reinterpret_cast<const Tin*>(buf + lane * g.pitch) + warp * KW;
      const float* wslice = wq + warp * KW;
      float2 ss2 = make_float2(0.f, 0.f);
      float2 dt2[S];
#pragma unroll
      for (int j = 0; j < S; ++j) dt2[j] = make_float2(0.f, 0.f);
      for (int kk = 0; kk < KW; kk += VEC) {
        float x[VEC];
        lds16(rowp + kk, x);  // one 16-byte load: 8 lanes per wavefront, no conflicts
#pragma unroll
        for (int q = 0; q < VEC; q += 2) ss2 = ffma2(make_float2(x[q], x[q + 1]), make_float2(x[q], x[q + 1]), ss2);
#pragma unroll
        for (int j = 0; j < S; ++j) {
#pragma unroll
          for (int q = 0; q < VEC; q += 4) {
            const float4 w4 = *reinterpret_cast<const float4*>(wslice + j * d + kk + q);
            dt2[j] = ffma2(make_float2(w4.x, w4.y), make_float2(x[q], x[q + 1]), dt2[j]);
            dt2[j] = ffma2(make_float2(w4.z, w4.w), make_float2(x[q + 2], x[q + 3]), dt2[j]);
          }
        }
      }
      float* rp = red + (warp * kMaxPairs + lane) * (S + 1);
      rp[0] = ss2.x + ss2.y;
#pragma unroll
      for (int j = 0; j < S; ++j) rp[1 + j] = dt2[j].x + dt2[j].y;
    }
    named_sync(1, kConsumers);

    // Scores e_ij = dot_ij / rms_i into alpha[r][i][j].
    for (int item = tid; item < P * S; item += kConsumers) {
      const int p = item / S, j = item - (item / S) * S;
      float ss = 0.f, dot = 0.f;
#pragma unroll
      for (int w = 0; w < kNW; ++w) {
        const float* rp = red + (w * kMaxPairs + p) * (S + 1);
        ss += rp[0];
        dot += rp[1 + j];
      }
      const int i = p / TM, r = p - (p / TM) * TM;
      alpha[(r * n + i) * S4 + j] = dot * rsqrtf(ss * inv_d + a.eps);
    }
    named_sync(1, kConsumers);

    // B. softmax over the n sources for each (row, query).
    for (int item = tid; item < TM * S; item += kConsumers) {
      const int r = item / S, j = item - (item / S) * S;
      float* e = alpha + r * n * S4 + j;
      float m = e[0];
      for (int i = 1; i < n; ++i) m = fmaxf(m, e[i * S4]);
      float z = 0.f;
      for (int i = 0; i < n; ++i) z += __expf(e[i * S4] - m);
      const float inv = 1.0f / z;
      for (int i = 0; i < n; ++i) e[i * S4] = __expf(e[i * S4] - m) * inv;
      if (a.lse && r < rows) a.lse[j * T + row0 + r] = m + __logf(z);
    }
    named_sync(1, kConsumers);

    // C. accumulate the S outputs of every row from the staged rows.
    for (int r = 0; r < rows; ++r) {
      float2 acc[S][CPT * 2];
#pragma unroll
      for (int j = 0; j < S; ++j)
#pragma unroll
        for (int q = 0; q < CPT * 2; ++q) acc[j][q] = make_float2(0.f, 0.f);
      for (int i = 0; i < n; ++i) {
        const Tin* rowp = reinterpret_cast<const Tin*>(buf + (i * TM + r) * g.pitch);
        const float* al = alpha + (r * n + i) * S4;
        float aw[S4];
#pragma unroll
        for (int j = 0; j < S4; j += 4) {
          const float4 a4 = *reinterpret_cast<const float4*>(al + j);
          aw[j] = a4.x; aw[j + 1] = a4.y; aw[j + 2] = a4.z; aw[j + 3] = a4.w;
        }
#pragma unroll
        for (int q = 0; q < CPT; ++q) {
          const int k = (tid + q * kConsumers) * 4;
          if (k < d) {
            float x[4];
            lds4(rowp + k, x);
#pragma unroll
            for (int j = 0; j < S; ++j) {
              const float2 a2 = make_float2(aw[j], aw[j]);
              acc[j][q * 2] = ffma2(a2, make_float2(x[0], x[1]), acc[j][q * 2]);
              acc[j][q * 2 + 1] = ffma2(a2, make_float2(x[2], x[3]), acc[j][q * 2 + 1]);
            }
          }
        }
      }
      const int64_t row = row0 + r;
#pragma unroll
      for (int q = 0; q < CPT; ++q) {
        const int k = (tid + q * kConsumers) * 4;
        if (k < d) {
#pragma unroll
          for (int j = 0; j < S; ++j) {
            const float o[4] = {acc[j][q * 2].x, acc[j][q * 2].y, acc[j][q * 2 + 1].x, acc[j][q * 2 + 1].y};
            st4(static_cast<Tin*>(a.out[j]) + row * d + k, o);
          }
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&empty_bar[b]));
    if (++b == 2) {
      b = 0;
      phase ^= 1u;
    }
  }
  if (!ok) atomicOr(&g_stage1_timeout, 1u);
}

template <typename Tin, int S>
cudaError_t launch_s(const MultiArgs& a, const Stage1Geom& g, cudaStream_t s) {
  const int cpt = (a.d / 4 + kConsumers - 1) / kConsumers;
  const void* fn = cpt == 1 ? reinterpret_cast<const void*>(&stage1_kernel<Tin, S, 1>)
                            : reinterpret_cast<const void*>(&stage1_kernel<Tin, S, 2>);
  cudaError_t e = allow_dynamic_smem(fn, g.total);
  if (e != cudaSuccess) return e;
  const int64_t tiles = (a.T + g.TM - 1) / g.TM;
  int64_t grid = sm_count();
  if (grid > tiles) grid = tiles;
  if (cpt == 1)
    return launch_pdl(stage1_kernel<Tin, S, 1>, static_cast<unsigned>(grid), kThreads, g.total, s, a, g);
  return launch_pdl(stage1_kernel<Tin, S, 2>, static_cast<unsigned>(grid), kThreads, g.total, s, a, g);
}

template <typename Tin>
cudaError_t launch_dtype(const MultiArgs& a, const Stage1Geom& g, cudaStream_t s) {
  switch (a.S) {
    case 1: return launch_s<Tin, 1>(a, g, s);
    case 2: return launch_s<Tin, 2>(a, g, s);
    case 3: return launch_s<Tin, 3>(a, g, s);
    case 4: return launch_s<Tin, 4>(a, g, s);
    case 5: return launch_s<Tin, 5>(a, g, s);
    case 6: return launch_s<Tin, 6>(a, g, s);
    case 7: return launch_s<Tin, 7>(a, g, s);
    case 8: return launch_s<Tin, 8>(a, g, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

// CUDA-core stage 1 (any storage dtype); the tensor-core kernel of
// stage1_tc.cu takes bf16 shapes it supports.
static bool stage1_cc_ok(const MultiArgs& a) {
  const int es = a.bf16 ? 2 : 4;
  const int vec = 16 / es;
  if (a.S < 1 || a.S > 8 || a.n_src < 1) return false;
  if (a.d % (kNW * vec) != 0 || a.d > 2048) return false;
  if (!aligned16(a.V) || !aligned16(a.W) || !aligned16(a.Gamma)) return false;
  if ((a.src_stride * es) % 16 != 0) return false;
  for (int j = 0; j < a.S; ++j)
    if (!aligned16(a.out[j])) return false;
  const Stage1Geom g = stage1_geom(a.n_src, a.d, a.S, es);
  return g.TM >= 1 && g.total <= kSmemLimit;
}

bool stage1_fast_ok(const MultiArgs& a) { return stage1_tc_ok(a) || stage1_cc_ok(a); }

cudaError_t launch_stage1_fast(const MultiArgs& a, cudaStream_t s) {
  if (stage1_tc_ok(a)) return launch_stage1_tc(a, s);
  const Stage1Geom g = stage1_geom(a.n_src, a.d, a.S, a.bf16 ? 2 : 4);
  return a.bf16 ? launch_dtype<bf16>(a, g, s) : launch_dtype<float>(a, g, s);
}

cudaError_t take_timeout_stage1(unsigned int* flag) {
  unsigned int zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(flag, g_stage1_timeout, sizeof(unsigned int));
  if (e != cudaSuccess) return e;
  return cudaMemcpyToSymbol(g_stage1_timeout, &zero, sizeof(unsigned int));
}

}  // namespace attnres
