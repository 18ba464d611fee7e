// Block AttnRes stage 1 with the scores on the tensor cores (bf16 storage).
//
// Same job as stage1.cu (datacamp explainer, "two-stage computation": the S
// pseudo-queries of a block against the cross-block sources, each source row
// read once): O_j[t] = sum_i softmax_i(e_ij) v_i[t], lse_j[t] = log sum_i
// exp(e_ij), e_ij = w_j^T RMSNorm_j(v_i[t]) (DepthBench reading notes section
// 2.3 / 2.5).
//
// The scores of a tile are a small dense contraction: with the tile's
// (source, row) pairs as the rows of A (16 x d, bf16, as staged) and the
// pseudo-queries as B (d x 8), e = A B / rms. It runs as warp-level m16n8k16
// MMAs: A comes from the staged rows with ldmatrix, and w * gamma (fp32) is
// split into bf16 hi + lo parts so the product keeps about 16 mantissa bits,
// accumulated in fp32. The sums of squares come from the same A fragments as
// the diagonal of A A^T (two more MMAs per step). The eight consumer warps
// split d; their partials meet in shared memory. The softmax over depth and
// the weighted accumulation of the S outputs (fp32 registers, packed fp32x2
// FMAs) run on the CUDA cores, as in stage1.cu. Rows arrive by per-row 1-D
// bulk copies into a padded pitch, double-buffered; two CTAs per SM overlap
// each other's barrier waits.
#include <math.h>
#include "common.cuh"
#include "internal.h"
namespace attnres {
namespace {
__device__ unsigned int g_stage1tc_timeout = 0;
constexpr int kNW = 8;                        // consumer warps
constexpr int kConsumers = kNW * kWarp;       // 256
constexpr int kThreads = kConsumers + kWarp;  // + producer warp
constexpr int kPairs = 16;                    // (source, row) pairs per tile: one m16 tile
constexpr int kQ = 8;                         // MMA query columns (queries >= S are zero)
constexpr int kBarBytes = 128;
struct TcGeom {
  int TM;          // rows per tile (kPairs / n)
  int pitch;       // bytes between staged rows (d * 2 + 16)
  int buf_bytes;   // one buffer: kPairs rows
  int w_off, red_off, alpha_off, buf_off, total;
};
inline int round_up(int x, int m) { return (x + m - 1) / m * m; }
inline TcGeom tc_geom(int n, int d, int S) {
  TcGeom g{};
  g.pitch = d * 2 + 16;
  g.TM = n > 0 ? kPairs / n : 0;
  g.w_off = kBarBytes;                      // bf16 hi rows [kQ], then lo rows [kQ]
  g.red_off = g.w_off + 2 * kQ * g.pitch;   // fp32 [kNW][kPairs][S+1] warp partials
  g.alpha_off = g.red_off + kNW * kPairs * (S + 1) * 4;
  g.buf_off = round_up(g.alpha_off + kPairs * round_up(S, 4) * 4, 128);
  g.buf_bytes = kPairs * g.pitch;
  g.total = g.buf_off + 2 * g.buf_bytes;
  return g;
}
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];" : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(addr));
}
__device__ __forceinline__ void mma16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3]) : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
template <int S, int CPT>
__global__ void __launch_bounds__(kThreads, CPT == 1 ? 2 : 1) stage1_tc_kernel(MultiArgs a, TcGeom g) {
  constexpr int S4 = (S + 3) / 4 * 4;
  extern __shared__ __align__(128) unsigned char smem[];
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem);
  uint64_t* empty_bar = full_bar + 2;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(full_bar + 4);
  unsigned char* wsm = smem + g.w_off;                          // w * gamma, bf16 hi / lo rows
  float* red = reinterpret_cast<float*>(smem + g.red_off);      // partial sums of squares / dots
  float* alpha = reinterpret_cast<float*>(smem + g.alpha_off);  // [TM][n][S4] scores, then weights
  unsigned char* bufs = smem + g.buf_off;                       // 2 tiles of staged rows
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int n = a.n_src, d = a.d, TM = g.TM;
  const int P = TM * n;
  const int64_t ntok = a.T;
  const int64_t ntiles_total = (ntok + TM - 1) / TM;
  const int64_t t0 = static_cast<int64_t>(blockIdx.x) * ntiles_total / gridDim.x;
  const int64_t t1 = static_cast<int64_t>(blockIdx.x + 1) * ntiles_total / gridDim.x;
  pdl_trigger();
  if (tid == 0) {
    for (int b = 0; b < 2; ++b) { mbar_init(smem_u32(&full_bar[b]), 1); mbar_init(smem_u32(&empty_bar[b]), kNW); }
    *reinterpret_cast<int*>(full_bar + 4) = 0;
    mbar_fence_init();
  }
  pdl_wait();
  // w * gamma as bf16 hi + lo rows (queries >= S are zero).
  for (int idx = tid; idx < kQ * d; idx += kThreads) {
    const int q = idx / d, k = idx - (idx / d) * d;
    const float w = q < S ? a.W[q * d + k] * a.Gamma[q * d + k] : 0.f;
    const bf16 hi = __float2bfloat16_rn(w);
    const bf16 lo = __float2bfloat16_rn(w - __bfloat162float(hi));
    reinterpret_cast<bf16*>(wsm + q * g.pitch)[k] = hi;
    reinterpret_cast<bf16*>(wsm + (kQ + q) * g.pitch)[k] = lo;
  }
  __syncthreads();
  if (warp == kNW) {
    // Producer: one bulk copy per (source, row) of the tile into a padded pitch.
    if (lane != 0) return;
    const char* src = static_cast<const char*>(a.V);
    const uint32_t row_bytes = static_cast<uint32_t>(d) * 2u;
    int b = 0; uint32_t phase = 0; int64_t issued = 0; bool ok = true;
    for (int64_t tile = t0; tile < t1; ++tile) {
      if (!mbar_wait(smem_u32(&empty_bar[b]), phase ^ 1u)) { ok = false; break; }
      const int64_t row0 = tile * TM;
      const int rows = static_cast<int>(min(static_cast<int64_t>(TM), ntok - row0));
      const uint32_t fb = smem_u32(&full_bar[b]);
      mbar_arrive_expect_tx(fb, row_bytes * rows * n);
      const uint32_t dst0 = smem_u32(bufs + b * g.buf_bytes);
      for (int i = 0; i < n; ++i)
        for (int r = 0; r < rows; ++r)
          bulk_g2s(dst0 + (i * TM + r) * g.pitch, src + (i * a.src_stride + (row0 + r) * d) * 2, row_bytes, fb);
      ++issued;
      if (++b == 2) { b = 0; phase ^= 1u; }
    }
    if (!ok) {
      atomicOr(&g_stage1tc_timeout, 1u);
      for (int64_t it = issued > 2 ? issued - 2 : 0; it < issued; ++it)
        (void)mbar_wait(smem_u32(&full_bar[it % 2]), static_cast<uint32_t>((it / 2) & 1));
    }
    return;
  }
  // Consumers.
  const float inv_d = 1.0f / static_cast<float>(d);
  const int KW = d / kNW;  // features of this warp's slice in the score pass
  const int a_row = (lane & 7) + ((lane >> 3) & 1) * 8;
  const int a_koff = (lane >> 4) * 8;
  const int b_row = (lane & 7) + ((lane >> 4) & 1) * kQ;
  const int b_koff = ((lane >> 3) & 1) * 8;
  const uint32_t b_base = smem_u32(wsm + b_row * g.pitch) + (warp * KW + b_koff) * 2;
  const int gid = lane >> 2, tig = lane & 3;
  int b = 0; uint32_t phase = 0; bool ok = true;
  for (int64_t tile = t0; tile < t1; ++tile) {
    // Giving up a wait is a joint decision (the consumers meet at barriers).
    if (!mbar_wait(smem_u32(&full_bar[b]), phase)) *abort_flag = 1;
    named_sync(1, kConsumers);
    if (*abort_flag) { ok = false; break; }
    const unsigned char* buf = bufs + b * g.buf_bytes;
    const int64_t row0 = tile * TM;
    const int rows = static_cast<int>(min(static_cast<int64_t>(TM), ntok - row0));
    // A. partial scores and sums of squares over this warp's slice (MMA).
    {
      const int pair = a_row < P ? a_row : 0;  // rows past P only pad the m16 tile
      const uint32_t a_base = smem_u32(buf + pair * g.pitch) + (warp * KW + a_koff) * 2;
      float sc[4] = {0.f, 0.f, 0.f, 0.f}, s0[4] = {0.f, 0.f, 0.f, 0.f}, s1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
      for (int k0 = 0; k0 < KW; k0 += 16) {
        uint32_t av[4], bv[4];
        ldsm_x4(a_base + k0 * 2, av);
        ldsm_x4(b_base + k0 * 2, bv);
        mma16816(sc, av, bv[0], bv[1]);  // hi part of w * gamma
        mma16816(sc, av, bv[2], bv[3]);  // lo part
        mma16816(s0, av, av[0], av[2]);  // A A^T, columns 0..7
        mma16816(s1, av, av[1], av[3]);  // A A^T, columns 8..15
      }
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int q = 2 * tig + e;
        if (q < S) {
          if (gid < P) red[(warp * kPairs + gid) * (S + 1) + 1 + q] = sc[e];
          if (gid + 8 < P) red[(warp * kPairs + gid + 8) * (S + 1) + 1 + q] = sc[2 + e];
        }
      }
      // Diagonal of A A^T: row gid in s0[gid & 1], row gid + 8 in s1[2 + (gid & 1)],
      // held by the lane whose 2 tig + e equals gid (selects keep registers).
      if (tig == (gid >> 1)) {
        const bool odd = gid & 1;
        if (gid < P) red[(warp * kPairs + gid) * (S + 1)] = odd ? s0[1] : s0[0];
        if (gid + 8 < P) red[(warp * kPairs + gid + 8) * (S + 1)] = odd ? s1[3] : s1[2];
      }
    }
    named_sync(1, kConsumers);
    // Scores e_ij = dot_ij / rms_i, summed over the warps' partials.
    for (int item = tid; item < P * S; item += kConsumers) {
      const int p = item / S, j = item - (item / S) * S;
      float ss = 0.f, dot = 0.f;
#pragma unroll
      for (int w = 0; w < kNW; ++w) { const float* rp = red + (w * kPairs + p) * (S + 1); ss += rp[0]; dot += rp[1 + j]; }
      const int i = p / TM, r = p - (p / TM) * TM;
      alpha[(r * n + i) * S4 + j] = dot * rsqrtf(ss * inv_d + a.eps);
    }
    named_sync(1, kConsumers);
    // B. softmax over the n sources for each (row, query): weights and lse.
    for (int item = tid; item < TM * S; item += kConsumers) {
      const int r = item / S, j = item - (item / S) * S;
      float* e = alpha + r * n * S4 + j;
      float m = e[0];
      for (int i = 1; i < n; ++i) m = fmaxf(m, e[i * S4]);
      float z = 0.f;
      for (int i = 0; i < n; ++i) z += __expf(e[i * S4] - m);
      const float inv = 1.0f / z;
      for (int i = 0; i < n; ++i) e[i * S4] = __expf(e[i * S4] - m) * inv;
      if (a.lse && r < rows) a.lse[j * ntok + row0 + r] = m + __logf(z);
    }
    named_sync(1, kConsumers);
    // C. the S outputs of every row from the staged rows (CUDA cores).
    for (int r = 0; r < rows; ++r) {
      float2 acc[S][CPT * 2];
#pragma unroll
      for (int j = 0; j < S; ++j)
#pragma unroll
        for (int q = 0; q < CPT * 2; ++q) acc[j][q] = make_float2(0.f, 0.f);
      for (int i = 0; i < n; ++i) {
        const bf16* rowp = reinterpret_cast<const bf16*>(buf + (i * TM + r) * g.pitch);
        const float* al = alpha + (r * n + i) * S4;
        float aw[S4];
#pragma unroll
        for (int j = 0; j < S4; j += 4) { const float4 a4 = *reinterpret_cast<const float4*>(al + j); aw[j] = a4.x; aw[j + 1] = a4.y; aw[j + 2] = a4.z; aw[j + 3] = a4.w; }
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
            st4(static_cast<bf16*>(a.out[j]) + row * d + k, o);
          }
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&empty_bar[b]));
    if (++b == 2) { b = 0; phase ^= 1u; }
  }
  if (!ok) atomicOr(&g_stage1tc_timeout, 1u);
}
template <int S, int CPT>
cudaError_t launch_sc(const MultiArgs& a, const TcGeom& g, cudaStream_t s) {
  auto k = stage1_tc_kernel<S, CPT>;
  cudaError_t e = allow_dynamic_smem(reinterpret_cast<const void*>(k), g.total);
  if (e != cudaSuccess) return e;
  const int64_t tiles = (a.T + g.TM - 1) / g.TM;
  int64_t grid = static_cast<int64_t>(sm_count()) * blocks_per_sm(reinterpret_cast<const void*>(k), kThreads, g.total);
  if (grid > tiles) grid = tiles;
  return launch_pdl(k, static_cast<unsigned>(grid), kThreads, g.total, s, a, g);
}
template <int S>
cudaError_t launch_s(const MultiArgs& a, const TcGeom& g, cudaStream_t s) {
  return (a.d / 4 <= kConsumers) ? launch_sc<S, 1>(a, g, s) : launch_sc<S, 2>(a, g, s);
}
}  // namespace
bool stage1_tc_ok(const MultiArgs& a) {
  if (!a.bf16 || a.S < 1 || a.S > 8 || a.n_src < 1 || a.n_src > kPairs) return false;
  if (a.d % (kNW * 16) != 0 || a.d > 2048) return false;
  if (!aligned16(a.V) || ((a.src_stride * 2) % 16) != 0) return false;
  for (int j = 0; j < a.S; ++j) if (!aligned16(a.out[j])) return false;
  return tc_geom(a.n_src, a.d, a.S).total <= 227 * 1024;
}
cudaError_t launch_stage1_tc(const MultiArgs& a, cudaStream_t s) {
  const TcGeom g = tc_geom(a.n_src, a.d, a.S);
  switch (a.S) {
    case 1: return launch_s<1>(a, g, s); case 2: return launch_s<2>(a, g, s);
    case 3: return launch_s<3>(a, g, s); case 4: return launch_s<4>(a, g, s);
    case 5: return launch_s<5>(a, g, s); case 6: return launch_s<6>(a, g, s);
    case 7: return launch_s<7>(a, g, s); case 8: return launch_s<8>(a, g, s);
    default: return cudaErrorInvalidValue;
  }
}
cudaError_t take_timeout_stage1tc(unsigned int* flag) {
  unsigned int zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(flag, g_stage1tc_timeout, sizeof(unsigned int));
  if (e != cudaSuccess) return e;
  return cudaMemcpyToSymbol(g_stage1tc_timeout, &zero, sizeof(unsigned int));
}
}  // namespace attnres
