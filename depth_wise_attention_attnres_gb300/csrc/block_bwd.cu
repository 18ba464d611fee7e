// The Block pass backward (attnres_block_bwd in api.cu drives these): the
// batched kernel below, which takes all S reads of a block in one pass, and
// the elementwise kernels of the per-read path, which runs the Full read's
// backward (full_bwd.cu) read by read for the other shapes.
//
// The Block pass reads, for sublayer k = n * S + j, the sources {embedding,
// b_1 .. b_n, P_k if j >= 1} (DepthBench reading notes section 2.5; LLMRes
// blog, "Block Attention Residuals"): b_m is the plain sum of block (m-1)'s
// outputs and P_k the sum of the earlier outputs of block n. By the chain rule
// the gradient of b_m reaches every member of block m-1 unchanged, and that of
// P_k every output of block n before k. The per-read path runs the reads in
// reverse order over fp32 copies of the sources; its kernels widen the
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

namespace attnres {
namespace {

// ------------------------------------------------ batched block backward --
//
// All S reads of block n in one pass over the tokens (d a multiple of 128 up
// to 1024, at most 8 cross-block sources and 8 sublayers per block). A CTA
// has d / 128 warps; warp w owns features 128 w .. 128 w + 127 (4 per lane)
// for every token, so the query-gradient sums du_j stay in its registers for
// the whole launch. A token's rows come into shared memory by cp.async: the
// next token's sources, outputs and dL/dout double-buffered, the token's own
// fp32 gradient rows fetched as it starts. Per token:
//  1. each lane reads its features of the block's sources X_0 .. X_n, the
//     running sums P_j (rebuilt from the outputs with the forward's fp32
//     additions) and dL/dout_j, and forms its parts of every dot product the
//     reads need: sum X_i^2, sum P_j^2, X_i . u_j, P_j . u_j, dz_j . X_i and
//     dz_j . P_j (u_j = w_j * gamma_j); the parts are summed over the warp by
//     a reduce-scatter of 32 values at a time and over the warps in shared
//     memory;
//  2. one thread per read forms its scores, softmax and score gradients, and
//     from them the coefficients of dX_i = sum_j (a_ij dz_j + r_i de_ij u_j)
//     - c_i X_i and of dP_j;
//  3. each lane forms its features of dX_i (added to the sources' gradient
//     rows), of dP_j, of du_j, and of every output's gradient dF_q = db +
//     sum_{j > q} dP_j, db being the gradient of this block's summary that
//     the later blocks accumulated.
constexpr int kBX = 8;              // cross-block sources at most (n + 1)
constexpr int kBQ = 8;              // sublayers (reads) per block at most
// Values reduced per token, for at most NX cross-block sources: [0, NX)
// sum X_i^2; then 8 sum P_j^2 (j >= 1); X_i.u_j at EX + NX j + i; dz_j.X_i at
// DaX + NX j + i; 8 P_j.u_j; 8 dz_j.P_j. Reduced 32 at a time.
template <int NX> struct BwdLayout {
  static constexpr int SsP = NX, EX = NX + kBQ, DaX = EX + kBQ * NX, EP = DaX + kBQ * NX, DaP = EP + kBQ;
  static constexpr int V = DaP + kBQ;
  static constexpr int Rounds = (V + 31) / 32;
};

__device__ __forceinline__ float dot4(const float (&a)[4], const float (&b)[4]) {
  return fmaf(a[0], b[0], fmaf(a[1], b[1], fmaf(a[2], b[2], a[3] * b[3])));
}

// Dynamic shared memory of the batched kernel: the next token's inputs
// (sources and outputs in T, dL/dout in TZ, double-buffered by cp.async) and
// the current token's fp32 gradient rows to update (sources', outputs', and
// the block summary's).
inline int64_t block_bwd_smem(const BlockBwdArgs& a) {
  const int n1 = a.N;  // sized for the largest block (n + 1 = N)
  const int64_t es = a.bf16 ? 2 : 4, zs = a.dz_bf16 ? 2 : 4;
  return 2 * static_cast<int64_t>(n1 + a.S - 1) * a.d * es + 2 * static_cast<int64_t>(a.S) * a.d * zs +
         static_cast<int64_t>(n1 + a.S + 1) * a.d * 4;
}

template <typename T, typename TZ, int NX>
__global__ void __launch_bounds__(1024 / 128 * 32, 1) block_bwd_batched_kernel(BlockBwdArgs a) {
  using Lay = BwdLayout<NX>;
  constexpr int kOffSsP = Lay::SsP, kOffEX = Lay::EX, kOffDaX = Lay::DaX, kOffEP = Lay::EP, kOffDaP = Lay::DaP;
  constexpr int kBV = Lay::Rounds * 32;
  extern __shared__ __align__(16) unsigned char bsm[];
  __shared__ float red[8][kBV];      // per-warp sums
  __shared__ float tot[kBV];         // CTA sums
  __shared__ float alpha[kBX][kBQ];  // coefficient of dz_j in dX_i
  __shared__ float beta[kBX][kBQ];   // coefficient of u_j in dX_i (r_i de_ij; also of X_i in du_j)
  __shared__ float ctmp[kBX][kBQ];   // de_ij e_ij r_i^2 / d, summed over j into cx[i]
  __shared__ float cx[kBX];
  __shared__ float pa[kBQ], pb[kBQ], pc[kBQ];  // the same for P_j (j >= 1)
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int W = blockDim.x >> 5;
  const int n1 = a.n + 1, S = a.S, d = a.d;
  const int k = warp * 128 + lane * 4;
  const int64_t k0 = static_cast<int64_t>(a.n) * S;
  const float inv_d = 1.0f / static_cast<float>(d);
  // u_j = w_j * gamma_j of this lane's features.
  float u[kBQ][4], du[kBQ][4];
#pragma unroll
  for (int j = 0; j < kBQ; ++j) {
    if (j < S) {
      float w4[4], g4[4];
      ldg4(a.W + (k0 + j) * d + k, w4);
      ldg4(a.Gamma + (k0 + j) * d + k, g4);
#pragma unroll
      for (int e = 0; e < 4; ++e) u[j][e] = w4[e] * g4[e];
    } else {
      u[j][0] = u[j][1] = u[j][2] = u[j][3] = 0.f;
    }
    du[j][0] = du[j][1] = du[j][2] = du[j][3] = 0.f;
  }
  const T* src = static_cast<const T*>(a.Src);
  const T* F = static_cast<const T*>(a.F);
  const TZ* dz = static_cast<const TZ*>(a.dOut);
  // Shared rows: inputs [2][rowsT][d] of T ([0, n1) sources, then the outputs
  // k0 .. k0 + S - 2), [2][S][d] of TZ, and the gradient rows [n1 + S + 1][d]
  // fp32 ([0, n1) the sources', then the outputs', then the summary's).
  const int rowsT = a.N + S - 1;  // buffer rows, sized for the largest block
  T* inT = reinterpret_cast<T*>(bsm);
  TZ* inZ = reinterpret_cast<TZ*>(bsm + 2 * static_cast<int64_t>(rowsT) * d * sizeof(T));
  float* gsm = reinterpret_cast<float*>(reinterpret_cast<unsigned char*>(inZ) + 2 * static_cast<int64_t>(S) * d * sizeof(TZ));
  const bool has_db = a.n + 1 < a.N;
  const int chT = d * static_cast<int>(sizeof(T)) / 16, chZ = d * static_cast<int>(sizeof(TZ)) / 16, chG = d / 4;
  // The CTA has d / 4 threads and a row has d * size / 16 chunks of 16 bytes,
  // a divisor of it: thread c copies chunk c % chunks of rows c / chunks,
  // c / chunks + threads / chunks, ...
  const int cT = threadIdx.x % chT, rT0 = threadIdx.x / chT, rTs = blockDim.x / chT;
  const int cZ = threadIdx.x % chZ, rZ0 = threadIdx.x / chZ, rZs = blockDim.x / chZ;
  const int cG = threadIdx.x % chG, rG0 = threadIdx.x / chG, rGs = blockDim.x / chG;
  auto issue_inputs = [&](int64_t t, int buf) {
    const uint32_t dT = smem_u32(inT + static_cast<int64_t>(buf) * rowsT * d) + cT * 16;
    for (int r = rT0; r < n1 + S - 1; r += rTs) {
      const T* g = r < n1 ? src + r * a.src_stride + t * d : F + (k0 + r - n1) * a.f_stride + t * d;
      cp_async16(dT + r * d * static_cast<int>(sizeof(T)), reinterpret_cast<const char*>(g) + cT * 16, true);
    }
    const uint32_t dZ = smem_u32(inZ + static_cast<int64_t>(buf) * S * d) + cZ * 16;
    for (int r = rZ0; r < S; r += rZs)
      cp_async16(dZ + r * d * static_cast<int>(sizeof(TZ)),
                 reinterpret_cast<const char*>(dz + (k0 + r) * a.dout_stride + t * d) + cZ * 16, true);
  };
  auto issue_grads = [&](int64_t t) {
    const uint32_t dG = smem_u32(gsm) + cG * 16;
    for (int r = rG0; r < n1 + S + (has_db ? 1 : 0); r += rGs) {
      const float* g = r < n1 ? a.dVs + r * a.E + t * d
                              : (r < n1 + S ? a.dF + (k0 + r - n1) * a.df_stride + t * d : a.dVs + (a.n + 1) * a.E + t * d);
      cp_async16(dG + r * d * 4, reinterpret_cast<const char*>(g) + cG * 16, true);
    }
  };
  int buf = 0;
  if (static_cast<int64_t>(blockIdx.x) < a.T) issue_inputs(blockIdx.x, 0);
  cp_async_commit();
  for (int64_t t = blockIdx.x; t < a.T; t += gridDim.x) {
    // This token's gradient rows, then the next token's inputs, in flight
    // while this token is worked on.
    issue_grads(t);
    cp_async_commit();
    if (t + gridDim.x < a.T) issue_inputs(t + gridDim.x, buf ^ 1);
    cp_async_commit();
    cp_async_wait<2>();
    __syncthreads();
    const T* xs = inT + static_cast<int64_t>(buf) * rowsT * d;
    const TZ* zsm = inZ + static_cast<int64_t>(buf) * S * d;
    // ---- 1. partial dot products of this lane's features
    float x[NX][4], p[kBQ][4], z[kBQ][4];
#pragma unroll
    for (int i = 0; i < NX; ++i) {
      if (i < n1) lds4(xs + i * d + k, x[i]);
      else x[i][0] = x[i][1] = x[i][2] = x[i][3] = 0.f;
    }
    p[0][0] = p[0][1] = p[0][2] = p[0][3] = 0.f;
#pragma unroll
    for (int j = 1; j < kBQ; ++j) {
      if (j < S) {
        float f[4];
        lds4(xs + (n1 + j - 1) * d + k, f);
#pragma unroll
        for (int e = 0; e < 4; ++e) p[j][e] = j == 1 ? f[e] : p[j - 1][e] + f[e];
      } else {
        p[j][0] = p[j][1] = p[j][2] = p[j][3] = 0.f;
      }
    }
#pragma unroll
    for (int j = 0; j < kBQ; ++j) {
      if (j < S) lds4(zsm + j * d + k, z[j]);
      else z[j][0] = z[j][1] = z[j][2] = z[j][3] = 0.f;
    }
#pragma unroll
    for (int r = 0; r < Lay::Rounds; ++r) {
      float v[32];
#pragma unroll
      for (int m = 0; m < 32; ++m) {
        const int idx = r * 32 + m;
        if (idx < kOffSsP) v[m] = dot4(x[idx], x[idx]);
        else if (idx < kOffEX) v[m] = dot4(p[idx - kOffSsP], p[idx - kOffSsP]);
        else if (idx < kOffDaX) v[m] = dot4(x[(idx - kOffEX) % NX], u[(idx - kOffEX) / NX]);
        else if (idx < kOffEP) v[m] = dot4(x[(idx - kOffDaX) % NX], z[(idx - kOffDaX) / NX]);
        else if (idx < kOffDaP) v[m] = dot4(p[idx - kOffEP], u[idx - kOffEP]);
        else if (idx < Lay::V) v[m] = dot4(p[idx - kOffDaP], z[idx - kOffDaP]);
        else v[m] = 0.f;
      }
      // Reduce-scatter over the warp: lane l ends with the warp's sum of v[l].
#pragma unroll
      for (int off = 16, h = 16; off >= 1; off >>= 1, h >>= 1) {
        const bool up = lane & off;
#pragma unroll
        for (int m = 0; m < 16; ++m)
          if (m < h) {
            const float send = up ? v[m] : v[m + h];
            const float keep = up ? v[m + h] : v[m];
            v[m] = keep + __shfl_xor_sync(0xffffffffu, send, off);
          }
      }
      red[warp][r * 32 + lane] = v[0];
    }
    __syncthreads();
    for (int i = threadIdx.x; i < kBV; i += blockDim.x) {
      float s = 0.f;
      for (int ww = 0; ww < W; ++ww) s += red[ww][i];
      tot[i] = s;
    }
    __syncthreads();
    // ---- 2. per read: scores, softmax, score gradients, coefficients
    if (threadIdx.x < S) {
      const int j = threadIdx.x;
      float rr[kBX], e[kBX], aa[kBX];
      float m = -INFINITY;
      for (int i = 0; i < n1; ++i) {
        rr[i] = rsqrtf(tot[i] * inv_d + a.eps);
        e[i] = rr[i] * tot[kOffEX + NX * j + i];
        m = fmaxf(m, e[i]);
      }
      float rP = 0.f, eP = 0.f;
      if (j >= 1) {
        rP = rsqrtf(tot[kOffSsP + j] * inv_d + a.eps);
        eP = rP * tot[kOffEP + j];
        m = fmaxf(m, eP);
      }
      float zs = 0.f;
      for (int i = 0; i < n1; ++i) {
        aa[i] = __expf(e[i] - m);
        zs += aa[i];
      }
      float aP = j >= 1 ? __expf(eP - m) : 0.f;
      zs += aP;
      const float inv = 1.0f / zs;
      float sda = 0.f;
      for (int i = 0; i < n1; ++i) {
        aa[i] *= inv;
        sda = fmaf(aa[i], tot[kOffDaX + NX * j + i], sda);
      }
      aP *= inv;
      if (j >= 1) sda = fmaf(aP, tot[kOffDaP + j], sda);
      for (int i = 0; i < n1; ++i) {
        const float de = aa[i] * (tot[kOffDaX + NX * j + i] - sda);
        alpha[i][j] = aa[i];
        beta[i][j] = rr[i] * de;
        ctmp[i][j] = de * e[i] * rr[i] * rr[i] * inv_d;
      }
      if (j >= 1) {
        const float deP = aP * (tot[kOffDaP + j] - sda);
        pa[j] = aP;
        pb[j] = rP * deP;
        pc[j] = deP * eP * rP * rP * inv_d;
      }
    }
    __syncthreads();
    if (threadIdx.x < n1) {
      float c = 0.f;
      for (int j = 0; j < S; ++j) c += ctmp[threadIdx.x][j];
      cx[threadIdx.x] = c;
    }
    cp_async_wait<1>();  // this token's gradient rows
    __syncthreads();
    // ---- 3. gradients of this lane's features
#pragma unroll
    for (int i = 0; i < NX; ++i) {
      if (i < n1) {
        float g[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) g[e] = -cx[i] * x[i][e];
#pragma unroll
        for (int j = 0; j < kBQ; ++j)
          if (j < S) {
            const float al = alpha[i][j], be = beta[i][j];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              g[e] = fmaf(al, z[j][e], fmaf(be, u[j][e], g[e]));
              du[j][e] = fmaf(be, x[i][e], du[j][e]);
            }
          }
        const float4 o = *reinterpret_cast<const float4*>(gsm + i * d + k);
        *reinterpret_cast<float4*>(a.dVs + i * a.E + t * d + k) =
            make_float4(o.x + g[0], o.y + g[1], o.z + g[2], o.w + g[3]);
      }
    }
    // dP_j and the outputs' gradients: dF_q += db + sum_{j > q} dP_j.
    float db[4] = {0.f, 0.f, 0.f, 0.f};
    if (has_db) lds4(gsm + (n1 + S) * d + k, db);
    float G[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int q = kBQ - 1; q >= 0; --q) {
      if (q >= S) continue;
      const float4 o = *reinterpret_cast<const float4*>(gsm + (n1 + q) * d + k);
      *reinterpret_cast<float4*>(a.dF + (k0 + q) * a.df_stride + t * d + k) =
          make_float4(o.x + db[0] + G[0], o.y + db[1] + G[1], o.z + db[2] + G[2], o.w + db[3] + G[3]);
      if (q >= 1) {
        const float c1 = pa[q], c2 = pb[q], c3 = pc[q];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          G[e] += fmaf(c1, z[q][e], fmaf(c2, u[q][e], -c3 * p[q][e]));
          du[q][e] = fmaf(c2, p[q][e], du[q][e]);
        }
      }
    }
    // The coefficient arrays and this buffer are rewritten by the next
    // token only after every thread has used them.
    __syncthreads();
    buf ^= 1;
  }
  cp_async_wait<0>();
  // dw_j += du_j * gamma_j, dgamma_j += du_j * w_j.
#pragma unroll
  for (int j = 0; j < kBQ; ++j) {
    if (j >= S) continue;
    float w4[4], g4[4];
    ldg4(a.W + (k0 + j) * d + k, w4);
    ldg4(a.Gamma + (k0 + j) * d + k, g4);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      if (a.dW) atomicAdd(a.dW + (k0 + j) * d + k + e, du[j][e] * g4[e]);
      if (a.dGamma) atomicAdd(a.dGamma + (k0 + j) * d + k + e, du[j][e] * w4[e]);
    }
  }
}

}  // namespace

bool block_bwd_batched_ok(const BlockBwdArgs& a) {
  if (a.d % 128 != 0 || a.d > 1024 || a.N > kBX || a.S > kBQ) return false;
  if (block_bwd_smem(a) > 200 * 1024) return false;
  const int es = a.bf16 ? 2 : 4, zs = a.dz_bf16 ? 2 : 4;
  return aligned16(a.Src) && aligned16(a.F) && aligned16(a.dOut) && aligned16(a.dVs) && aligned16(a.dF) &&
         aligned16(a.W) && aligned16(a.Gamma) && (a.src_stride * es) % 16 == 0 && (a.f_stride * es) % 16 == 0 &&
         (a.dout_stride * zs) % 16 == 0 && (a.df_stride * 4) % 16 == 0;
}

namespace {

template <int NX>
cudaError_t launch_block_bwd_nx(const BlockBwdArgs& a, cudaStream_t s) {
  const int threads = a.d / 128 * 32;
  const void* fn = a.bf16 ? (a.dz_bf16 ? reinterpret_cast<const void*>(&block_bwd_batched_kernel<bf16, bf16, NX>)
                                       : reinterpret_cast<const void*>(&block_bwd_batched_kernel<bf16, float, NX>))
                          : (a.dz_bf16 ? reinterpret_cast<const void*>(&block_bwd_batched_kernel<float, bf16, NX>)
                                       : reinterpret_cast<const void*>(&block_bwd_batched_kernel<float, float, NX>));
  const int smem = static_cast<int>(block_bwd_smem(a));
  cudaError_t e = allow_dynamic_smem(fn, smem);
  if (e != cudaSuccess) return e;
  int64_t grid = static_cast<int64_t>(sm_count()) * blocks_per_sm(fn, threads, smem);
  if (grid > a.T) grid = a.T;
  const unsigned g = static_cast<unsigned>(grid > 0 ? grid : 1);
  if (a.bf16) {
    if (a.dz_bf16) block_bwd_batched_kernel<bf16, bf16, NX><<<g, threads, smem, s>>>(a);
    else block_bwd_batched_kernel<bf16, float, NX><<<g, threads, smem, s>>>(a);
  } else {
    if (a.dz_bf16) block_bwd_batched_kernel<float, bf16, NX><<<g, threads, smem, s>>>(a);
    else block_bwd_batched_kernel<float, float, NX><<<g, threads, smem, s>>>(a);
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_block_bwd_batched(const BlockBwdArgs& a, cudaStream_t s) {
  const int n1 = a.n + 1;
  return n1 <= 2 ? launch_block_bwd_nx<2>(a, s) : n1 <= 4 ? launch_block_bwd_nx<4>(a, s) : launch_block_bwd_nx<8>(a, s);
}

}  // namespace attnres
