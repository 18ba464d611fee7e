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
// the whole launch. A token's rows come into shared memory on the TMA engine,
// issued by the last warp and signalled on mbarriers: the next token's
// sources, outputs and dL/dout (double-buffered, one bulk copy per row,
// issued while the per-read step runs), and the token's own fp32 gradient
// rows (two tensor copies as it starts). Per token:
//  1. each lane reads its features of the block's sources X_0 .. X_n, the
//     running sums P_j (rebuilt from the outputs with the forward's fp32
//     additions) and dL/dout_j, and forms its parts of every dot product the
//     reads need: sum X_i^2, sum P_j^2, X_i . u_j, P_j . u_j, dz_j . X_i and
//     dz_j . P_j (u_j = w_j * gamma_j); the parts are summed over the warp by
//     a reduce-scatter of 32 values at a time and over the warps in shared
//     memory;
//  2. a group of 16 lanes per read forms its scores, softmax and score
//     gradients (one source a lane, sums by shuffles), and from them the
//     coefficients of dX_i = sum_j (a_ij dz_j + r_i de_ij u_j) - c_i X_i and
//     of dP_j;
//  3. each lane forms its features of dX_i (added to the sources' gradient
//     rows), of dP_j, of du_j, and of every output's gradient dF_q = db +
//     sum_{j > q} dP_j, db being the gradient of this block's summary that
//     the later blocks accumulated.
// With bf16 rows and bf16 dL/dout (the TC instance), step 1 runs on the
// tensor cores instead: the token's staged rows R (the sources, then the
// outputs k0 .. k0 + S - 2; at most 15, padded to 16) are the A operand of
// mma.sync m16n8k16 over the warp's 128 features, and the B operands are R
// itself (its Gram matrix; the B fragments are the A fragments), u_j split
// into three bf16 parts (hi + mid + lo = u_j to fp32 accuracy, so the scores
// keep fp32 accuracy), and dL/dout_j. Every product of stored bf16 values is
// exact in fp32. The dot products with the running sums follow by linearity:
// P_j . y = sum_{m < j} F_m . y. The 16 x 32 partial matrix of each warp is
// summed over the warps in shared memory.
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
// TC instance: the reduced matrix is R . [R | u | dz], 16 rows of 32 columns
// (0-15 the Gram matrix, 16-23 R . u_j, 24-31 R . dz_j). A warp's partials
// are stored with rows 40 floats apart, so its fragment stores hit distinct
// banks; the CTA sums with rows 33 apart, so the lanes of a read's group,
// one row each, do too.
constexpr int kTcCols = 32, kTcLd = 40, kTcTot = 33;

// Shared-memory row strides (elements): 16 bytes of padding, so the eight
// 16-byte rows one ldmatrix reads fall in distinct banks.
inline __host__ __device__ int padded_ld(int d, int elem_bytes) { return d + 16 / elem_bytes; }

// x = hi + mid + lo, each a bf16: hi and mid are taken from the exact
// remainders, so the sum is x to within a rounding of lo (about 2^-27 |x|).
__device__ __forceinline__ void split3_bf16(float x, float& hi, float& mid, float& lo) {
  hi = __bfloat162float(__float2bfloat16_rn(x));
  const float r = x - hi;
  mid = __bfloat162float(__float2bfloat16_rn(r));
  lo = r - mid;
}

__device__ __forceinline__ float dot4(const float (&a)[4], const float (&b)[4]) {
  return fmaf(a[0], b[0], fmaf(a[1], b[1], fmaf(a[2], b[2], a[3] * b[3])));
}

// Dynamic shared memory of the batched kernel: the next token's inputs
// (sources and outputs in T, dL/dout in TZ, double-buffered, rows padded)
// and the current token's fp32 gradient rows to update (sources', the block
// summary's, outputs'), 128-byte aligned.
inline int64_t block_bwd_smem(const BlockBwdArgs& a) {
  const int n1 = a.N;  // sized for the largest block (n + 1 = N)
  const int es = a.bf16 ? 2 : 4, zs = a.dz_bf16 ? 2 : 4;
  return 2 * static_cast<int64_t>(n1 + a.S - 1) * padded_ld(a.d, es) * es +
         2 * static_cast<int64_t>(a.S) * padded_ld(a.d, zs) * zs + 128 +  // the gradient rows start 128-aligned
         static_cast<int64_t>(n1 + a.S + 1) * a.d * 4;
}

// The gradient rows as 4-d fp32 tensors (feature within a chunk of 128,
// chunk, token, row), each box one token's rows whole: the scratch's rows
// 0 .. n (the block's sources) and n + 1 (the summary block n makes, when
// there is one), and dF's rows n S .. n S + S - 1.
bool encode_grad_maps(const BlockBwdArgs& a, CUtensorMap* mv, CUtensorMap* mf) {
  PFN_cuTensorMapEncodeTiled_v12000 fn = tensor_map_encode_fn();
  if (!fn) return false;
  const int n1 = a.n + 1, rv = n1 + (a.n + 1 < a.N ? 1 : 0);
  const int64_t L = static_cast<int64_t>(a.N) * a.S;
  const cuuint32_t es[4] = {1, 1, 1, 1};
  const cuuint64_t dv[4] = {128, static_cast<cuuint64_t>(a.d / 128), static_cast<cuuint64_t>(a.T),
                            static_cast<cuuint64_t>(a.N)};
  const cuuint64_t sv[3] = {512, static_cast<cuuint64_t>(a.d) * 4, static_cast<cuuint64_t>(a.E) * 4};
  const cuuint32_t bv[4] = {128, static_cast<cuuint32_t>(a.d / 128), 1, static_cast<cuuint32_t>(rv)};
  if (fn(mv, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, a.dVs, dv, sv, bv, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
         CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return false;
  const cuuint64_t df[4] = {128, static_cast<cuuint64_t>(a.d / 128), static_cast<cuuint64_t>(a.T),
                            static_cast<cuuint64_t>(L)};
  const cuuint64_t sf[3] = {512, static_cast<cuuint64_t>(a.d) * 4,
                            static_cast<cuuint64_t>(L > 1 ? a.df_stride : a.E) * 4};
  const cuuint32_t bf[4] = {128, static_cast<cuuint32_t>(a.d / 128), 1, static_cast<cuuint32_t>(a.S)};
  return fn(mf, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, a.dF, df, sf, bf, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

// One token's rows of a gradient map into shared memory (128-byte aligned).
__device__ __forceinline__ void tma_load_rows(uint32_t dst, const CUtensorMap* map, int tok, int row0, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, "
      "%5}], [%6];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(0), "r"(0), "r"(tok), "r"(row0), "r"(bar)
      : "memory");
}

__device__ unsigned int g_blockbwd_timeout = 0;

template <typename T, typename TZ, int NX, bool TC>
__global__ void __launch_bounds__(1024 / 128 * 32, 1)
    block_bwd_batched_kernel(BlockBwdArgs a, const __grid_constant__ CUtensorMap gmv,
                             const __grid_constant__ CUtensorMap gmf) {
  static_assert(!TC || (sizeof(T) == 2 && sizeof(TZ) == 2), "the tensor-core instance takes bf16 rows");
  using Lay = BwdLayout<NX>;
  constexpr int kOffSsP = Lay::SsP, kOffEX = Lay::EX, kOffDaX = Lay::DaX, kOffEP = Lay::EP, kOffDaP = Lay::DaP;
  constexpr int kBV = Lay::Rounds * 32;
  constexpr int kRedW = TC ? 16 * kTcLd : kBV, kTot = TC ? 16 * kTcCols : kBV;
  constexpr int kTotSize = TC ? 16 * kTcTot : kBV;
  extern __shared__ __align__(16) unsigned char bsm[];
  __shared__ __align__(16) float red[8][kRedW];  // per-warp sums
  __shared__ float tot[kTotSize];                // CTA sums
  // Coefficients, rows padded (12 and 9 floats) so the per-read step's
  // writes, one source row a lane, hit distinct banks.
  __shared__ __align__(16) float alpha[kBX][kBQ + 4];  // coefficient of dz_j in dX_i
  __shared__ __align__(16) float beta[kBX][kBQ + 4];   // coefficient of u_j in dX_i (r_i de_ij; also of X_i in du_j)
  __shared__ float ctmp[kBX][kBQ + 1];                 // de_ij e_ij r_i^2 / d, summed over j into cx[i]
  __shared__ float cx[kBX];
  __shared__ __align__(16) float pa[kBQ];  // the same for P_j (j >= 1)
  __shared__ __align__(16) float pb[kBQ];
  __shared__ __align__(16) float pc[kBQ];
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
  // TC: B fragments of u_j (j = lane / 4) over the warp's 8 k-steps of 16
  // features, in three bf16 parts.
  uint32_t ufr[3][8][2];
  if constexpr (TC) {
    const int gj = lane >> 2, t4 = lane & 3;
#pragma unroll
    for (int ks = 0; ks < 8; ++ks)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int f = warp * 128 + ks * 16 + h * 8 + 2 * t4;
        float u0 = 0.f, u1 = 0.f;
        if (gj < S) {
          const float2 w2 = *reinterpret_cast<const float2*>(a.W + (k0 + gj) * d + f);
          const float2 m2 = *reinterpret_cast<const float2*>(a.Gamma + (k0 + gj) * d + f);
          u0 = w2.x * m2.x;
          u1 = w2.y * m2.y;
        }
        float h0, m0, l0, h1, m1, l1;
        split3_bf16(u0, h0, m0, l0);
        split3_bf16(u1, h1, m1, l1);
        ufr[0][ks][h] = pack_bf16x2(h0, h1);
        ufr[1][ks][h] = pack_bf16x2(m0, m1);
        ufr[2][ks][h] = pack_bf16x2(l0, l1);
      }
  }
  const T* src = static_cast<const T*>(a.Src);
  const T* F = static_cast<const T*>(a.F);
  const TZ* dz = static_cast<const TZ*>(a.dOut);
  // Shared rows: inputs [2][rowsT][ldT] of T ([0, n1) sources, then the
  // outputs k0 .. k0 + S - 2), [2][S][ldZ] of TZ, and the gradient rows
  // [n1 + S + 1][d] fp32 ([0, n1) the sources', n1 the summary's, then the
  // outputs'), 128-byte aligned for the tensor copies.
  const int rowsT = a.N + S - 1;  // buffer rows, sized for the largest block
  const int ldT = padded_ld(d, sizeof(T)), ldZ = padded_ld(d, sizeof(TZ));
  T* inT = reinterpret_cast<T*>(bsm);
  TZ* inZ = reinterpret_cast<TZ*>(bsm + 2 * static_cast<int64_t>(rowsT) * ldT * sizeof(T));
  unsigned char* gbase = reinterpret_cast<unsigned char*>(inZ) + 2 * static_cast<int64_t>(S) * ldZ * sizeof(TZ);
  float* gsm = reinterpret_cast<float*>(gbase + ((128u - (smem_u32(gbase) & 127u)) & 127u));
  const bool has_db = a.n + 1 < a.N;
  // Rows move on the TMA engine, issued by the CTA's last warp: the inputs
  // by bulk copies, one row per lane, each lane arriving on the buffer's
  // mbarrier with its byte count (bars[0] and bars[1]: n1 + S - 1 rows of T,
  // S of TZ); the gradient rows by two tensor copies from lane 0 (bars[2]).
  __shared__ __align__(8) uint64_t bars[3];
  const bool issuer = warp == W - 1;
  const int in_rows = n1 + S - 1 + S, g_rows = n1 + S + (has_db ? 1 : 0);  // at most 23 and 17
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bars[0]), in_rows);
    mbar_init(smem_u32(&bars[1]), in_rows);
    mbar_init(smem_u32(&bars[2]), 1);
    mbar_fence_init();
  }
  __syncthreads();
  auto issue_inputs = [&](int64_t t, int b) {
    const int r = lane;
    if (r >= in_rows) return;
    const uint32_t bar = smem_u32(&bars[b]);
    if (r < n1 + S - 1) {
      const T* g = r < n1 ? src + r * a.src_stride + t * d : F + (k0 + r - n1) * a.f_stride + t * d;
      mbar_arrive_expect_tx(bar, d * sizeof(T));
      bulk_g2s(smem_u32(inT + (static_cast<int64_t>(b) * rowsT + r) * ldT), g, d * sizeof(T), bar);
    } else {
      const int q = r - (n1 + S - 1);
      mbar_arrive_expect_tx(bar, d * sizeof(TZ));
      bulk_g2s(smem_u32(inZ + (static_cast<int64_t>(b) * S + q) * ldZ), dz + (k0 + q) * a.dout_stride + t * d,
               d * sizeof(TZ), bar);
    }
  };
  auto issue_grads = [&](int64_t t) {
    if (lane != 0) return;
    const uint32_t bar = smem_u32(&bars[2]);
    mbar_arrive_expect_tx(bar, static_cast<uint32_t>(g_rows * d * 4));
    tma_load_rows(smem_u32(gsm), &gmv, static_cast<int>(t), 0, bar);
    tma_load_rows(smem_u32(gsm + (n1 + 1) * d), &gmf, static_cast<int>(t), static_cast<int>(k0), bar);
  };
  // Every thread tracks the barriers' parities and which copies are pending
  // (the issuer waits for those before it leaves after a timeout).
  uint32_t ph0 = 0, ph1 = 0, phg = 0;
  bool pend0 = false, pend1 = false, pendg = false, timed_out = false;
  int buf = 0;
  if (static_cast<int64_t>(blockIdx.x) < a.T) {
    if (issuer) issue_inputs(blockIdx.x, 0);
    pend0 = true;
  }
  for (int64_t t = blockIdx.x; t < a.T; t += gridDim.x) {
    // This token's gradient rows (the previous token's are consumed: every
    // thread passed the barrier that ends its iteration).
    if (issuer) issue_grads(t);
    pendg = true;
    {
      const bool ok = mbar_wait(smem_u32(&bars[buf]), buf ? ph1 : ph0);
      if (__syncthreads_or(!ok)) {
        timed_out = true;
        break;
      }
      if (buf) { ph1 ^= 1u; pend1 = false; } else { ph0 ^= 1u; pend0 = false; }
    }
    const T* xs = inT + static_cast<int64_t>(buf) * rowsT * ldT;
    const TZ* zsm = inZ + static_cast<int64_t>(buf) * S * ldZ;
    // This lane's features of the sources, the running sums (the forward's
    // fp32 additions) and dL/dout.
    float x[NX][4], p[kBQ][4], z[kBQ][4];
    auto load_x = [&]() {
#pragma unroll
      for (int i = 0; i < NX; ++i) {
        if (i < n1) lds4(xs + i * ldT + k, x[i]);
        else x[i][0] = x[i][1] = x[i][2] = x[i][3] = 0.f;
      }
    };
    auto load_p = [&]() {
      p[0][0] = p[0][1] = p[0][2] = p[0][3] = 0.f;
#pragma unroll
      for (int j = 1; j < kBQ; ++j) {
        if (j < S) {
          float f[4];
          lds4(xs + (n1 + j - 1) * ldT + k, f);
#pragma unroll
          for (int e = 0; e < 4; ++e) p[j][e] = j == 1 ? f[e] : p[j - 1][e] + f[e];
        } else {
          p[j][0] = p[j][1] = p[j][2] = p[j][3] = 0.f;
        }
      }
    };
    auto load_z = [&]() {
#pragma unroll
      for (int j = 0; j < kBQ; ++j) {
        if (j < S) lds4(zsm + j * ldZ + k, z[j]);
        else z[j][0] = z[j][1] = z[j][2] = z[j][3] = 0.f;
      }
    };
    // ---- 1. partial dot products of this warp's features
    if constexpr (TC) {
      const int gj = lane >> 2, t4 = lane & 3;
      // ldmatrix row addresses: A rows (lane & 7) + (lane & 8), k offset
      // 8 (lane >> 4); dz rows lane & 7, k offset lane & 8. Rows past the
      // block's last are clamped to it (their products are not used).
      const int rmax = n1 + S - 2;
      const uint32_t aA = smem_u32(xs + min((lane & 7) + (lane & 8), rmax) * ldT + warp * 128 + (lane >> 4) * 8);
      const uint32_t aZ = smem_u32(zsm + min(lane & 7, S - 1) * ldZ + warp * 128 + (lane & 8));
      float cg0[4] = {0.f, 0.f, 0.f, 0.f}, cg1[4] = {0.f, 0.f, 0.f, 0.f}, cz[4] = {0.f, 0.f, 0.f, 0.f};
      float cu0[4] = {0.f, 0.f, 0.f, 0.f}, cu1[4] = {0.f, 0.f, 0.f, 0.f}, cu2[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        uint32_t fa[4], z0, z1;
        ldsm_x4(aA + ks * 32, fa);
        ldsm_x2(aZ + ks * 32, z0, z1);
        mma16816(cg0, fa, fa[0], fa[2]);  // R . R_c, c = 0..7
        mma16816(cg1, fa, fa[1], fa[3]);  // R . R_c, c = 8..15
        mma16816(cu0, fa, ufr[0][ks][0], ufr[0][ks][1]);
        mma16816(cu1, fa, ufr[1][ks][0], ufr[1][ks][1]);
        mma16816(cu2, fa, ufr[2][ks][0], ufr[2][ks][1]);
        mma16816(cz, fa, z0, z1);
      }
      float cu[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) cu[e] = (cu0[e] + cu1[e]) + cu2[e];
      // Accumulator fragment: rows gj and gj + 8, columns 2 t4 and 2 t4 + 1.
      float* rw = red[warp];
      auto put = [&](int col, const float (&c)[4]) {
        *reinterpret_cast<float2*>(rw + gj * kTcLd + col + 2 * t4) = make_float2(c[0], c[1]);
        *reinterpret_cast<float2*>(rw + (gj + 8) * kTcLd + col + 2 * t4) = make_float2(c[2], c[3]);
      };
      put(0, cg0);
      put(8, cg1);
      put(16, cu);
      put(24, cz);
    } else {
    load_x();
    load_p();
    load_z();
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
    }
    __syncthreads();
    for (int i = threadIdx.x; i < kTot; i += blockDim.x) {
      const int ri = TC ? (i >> 5) * kTcLd + (i & 31) : i;
      float s = 0.f;
      for (int ww = 0; ww < W; ++ww) s += red[ww][ri];
      tot[TC ? (i >> 5) * kTcTot + (i & 31) : i] = s;
    }
    __syncthreads();
    // The next token's inputs, issued while the per-read step runs; their
    // buffer was last read in the previous iteration.
    if (t + gridDim.x < a.T) {
      if (issuer) issue_inputs(t + gridDim.x, buf ^ 1);
      if (buf) pend0 = true; else pend1 = true;
    }
    // The reduced dot products of the sources: sum X_i^2, X_i . u_j, dz_j . X_i.
    auto ssx = [&](int i) { return TC ? tot[i * (kTcTot + 1)] : tot[i]; };
    auto ex = [&](int i, int j) { return TC ? tot[i * kTcTot + 16 + j] : tot[kOffEX + NX * j + i]; };
    auto dax = [&](int i, int j) { return TC ? tot[i * kTcTot + 24 + j] : tot[kOffDaX + NX * j + i]; };
    // ---- 2. per read: scores, softmax, score gradients, coefficients. Read
    // j goes to a group of 16 lanes: lane i < n1 takes source i, lane n1 the
    // running sum (j >= 1); the softmax sums run over the group by shuffles.
    {
      const int gl = threadIdx.x & 15;
      const unsigned gmask = 0xffffu << (threadIdx.x & 16);
      for (int j = threadIdx.x >> 4; j < S; j += blockDim.x >> 4) {
        const bool xl = gl < n1, pl = gl == n1 && j >= 1;
        // The running sum's: sum P_j^2, P_j . u_j, dz_j . P_j. TC: by
        // linearity from the output rows, P_j . y = sum_{m < j} F_m . y, one
        // row m a lane, summed over the group.
        float ssp = 0.f, ep = 0.f, dap = 0.f;
        if constexpr (TC) {
          if (gl < j) {
            const float* row = tot + (n1 + gl) * kTcTot;
#pragma unroll
            for (int m2 = 0; m2 < kBQ - 1; ++m2)
              if (m2 < j) ssp += row[n1 + m2];
            ep = row[16 + j];
            dap = row[24 + j];
          }
#pragma unroll
          for (int o = 8; o; o >>= 1) {
            ssp += __shfl_xor_sync(gmask, ssp, o);
            ep += __shfl_xor_sync(gmask, ep, o);
            dap += __shfl_xor_sync(gmask, dap, o);
          }
        } else if (pl) {
          ssp = tot[kOffSsP + j];
          ep = tot[kOffEP + j];
          dap = tot[kOffDaP + j];
        }
        float rr = 0.f, e = -INFINITY, da = 0.f;
        if (xl) {
          rr = rsqrtf(ssx(gl) * inv_d + a.eps);
          e = rr * ex(gl, j);
          da = dax(gl, j);
        } else if (pl) {
          rr = rsqrtf(ssp * inv_d + a.eps);
          e = rr * ep;
          da = dap;
        }
        float m = e;
#pragma unroll
        for (int o = 8; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(gmask, m, o));
        float al = (xl || pl) ? __expf(e - m) : 0.f;
        float zs = al;
#pragma unroll
        for (int o = 8; o; o >>= 1) zs += __shfl_xor_sync(gmask, zs, o);
        al *= 1.0f / zs;
        float sda = al * da;
#pragma unroll
        for (int o = 8; o; o >>= 1) sda += __shfl_xor_sync(gmask, sda, o);
        const float de = al * (da - sda);
        if (xl) {
          alpha[gl][j] = al;
          beta[gl][j] = rr * de;
          ctmp[gl][j] = de * e * rr * rr * inv_d;
        } else if (pl) {
          pa[j] = al;
          pb[j] = rr * de;
          pc[j] = de * e * rr * rr * inv_d;
        }
      }
    }
    __syncthreads();
    if (threadIdx.x < n1) {
      float c = 0.f;
      for (int j = 0; j < S; ++j) c += ctmp[threadIdx.x][j];
      cx[threadIdx.x] = c;
    }
    {  // this token's gradient rows
      const bool ok = mbar_wait(smem_u32(&bars[2]), phg);
      if (__syncthreads_or(!ok)) {
        timed_out = true;
        break;
      }
      phg ^= 1u;
      pendg = false;
    }
    // ---- 3. gradients of this lane's features
    // (TC: dL/dout here, the sources' rows one at a time below, the running
    // sums after them.)
    if constexpr (TC) load_z();
#pragma unroll
    for (int i = 0; i < NX; ++i) {
      if (i < n1) {
        if constexpr (TC) lds4(xs + i * ldT + k, x[i]);
        // Packed fp32x2 FMAs (each half an ordinary fused multiply-add).
        float al8[kBQ], be8[kBQ];
        *reinterpret_cast<float4*>(al8) = *reinterpret_cast<const float4*>(&alpha[i][0]);
        *reinterpret_cast<float4*>(al8 + 4) = *reinterpret_cast<const float4*>(&alpha[i][4]);
        *reinterpret_cast<float4*>(be8) = *reinterpret_cast<const float4*>(&beta[i][0]);
        *reinterpret_cast<float4*>(be8 + 4) = *reinterpret_cast<const float4*>(&beta[i][4]);
        const float ncx = -cx[i];
        const float2 x01 = make_float2(x[i][0], x[i][1]), x23 = make_float2(x[i][2], x[i][3]);
        float2 g01 = make_float2(ncx * x[i][0], ncx * x[i][1]), g23 = make_float2(ncx * x[i][2], ncx * x[i][3]);
#pragma unroll
        for (int j = 0; j < kBQ; ++j)
          if (j < S) {
            const float2 al = make_float2(al8[j], al8[j]), be = make_float2(be8[j], be8[j]);
            g01 = ffma2(al, make_float2(z[j][0], z[j][1]), ffma2(be, make_float2(u[j][0], u[j][1]), g01));
            g23 = ffma2(al, make_float2(z[j][2], z[j][3]), ffma2(be, make_float2(u[j][2], u[j][3]), g23));
            const float2 d01 = ffma2(be, x01, make_float2(du[j][0], du[j][1]));
            const float2 d23 = ffma2(be, x23, make_float2(du[j][2], du[j][3]));
            du[j][0] = d01.x; du[j][1] = d01.y; du[j][2] = d23.x; du[j][3] = d23.y;
          }
        const float4 o = *reinterpret_cast<const float4*>(gsm + i * d + k);
        *reinterpret_cast<float4*>(a.dVs + i * a.E + t * d + k) =
            make_float4(o.x + g01.x, o.y + g01.y, o.z + g23.x, o.w + g23.y);
      }
    }
    // dP_j and the outputs' gradients: dF_q += db + sum_{j > q} dP_j.
    if constexpr (TC) load_p();
    float db[4] = {0.f, 0.f, 0.f, 0.f};
    if (has_db) lds4(gsm + n1 * d + k, db);
    float G[4] = {0.f, 0.f, 0.f, 0.f};
    float pa8[kBQ], pb8[kBQ], pc8[kBQ];
#pragma unroll
    for (int h = 0; h < kBQ; h += 4) {
      *reinterpret_cast<float4*>(pa8 + h) = *reinterpret_cast<const float4*>(pa + h);
      *reinterpret_cast<float4*>(pb8 + h) = *reinterpret_cast<const float4*>(pb + h);
      *reinterpret_cast<float4*>(pc8 + h) = *reinterpret_cast<const float4*>(pc + h);
    }
#pragma unroll
    for (int q = kBQ - 1; q >= 0; --q) {
      if (q >= S) continue;
      const float4 o = *reinterpret_cast<const float4*>(gsm + (n1 + 1 + q) * d + k);
      *reinterpret_cast<float4*>(a.dF + (k0 + q) * a.df_stride + t * d + k) =
          make_float4(o.x + db[0] + G[0], o.y + db[1] + G[1], o.z + db[2] + G[2], o.w + db[3] + G[3]);
      if (q >= 1) {
        const float c1 = pa8[q], c2 = pb8[q], c3 = pc8[q];
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
  if (timed_out) {
    // Wait (bounded) for the copies still in flight into shared memory, then
    // report and stop.
    if (threadIdx.x == blockDim.x - 1) {
      if (pend0) (void)mbar_wait(smem_u32(&bars[0]), ph0);
      if (pend1) (void)mbar_wait(smem_u32(&bars[1]), ph1);
      if (pendg) (void)mbar_wait(smem_u32(&bars[2]), phg);
      atomicOr(&g_blockbwd_timeout, 1u);
    }
    return;
  }
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
  if (a.d % 128 != 0 || a.d > 1024 || a.N > kBX || a.S > kBQ || a.T > INT32_MAX) return false;
  if (tensor_map_encode_fn() == nullptr) return false;
  if (block_bwd_smem(a) > 200 * 1024) return false;
  const int es = a.bf16 ? 2 : 4, zs = a.dz_bf16 ? 2 : 4;
  return aligned16(a.Src) && aligned16(a.F) && aligned16(a.dOut) && aligned16(a.dVs) && aligned16(a.dF) &&
         aligned16(a.W) && aligned16(a.Gamma) && (a.src_stride * es) % 16 == 0 && (a.f_stride * es) % 16 == 0 &&
         (a.dout_stride * zs) % 16 == 0 && (a.df_stride * 4) % 16 == 0;
}

namespace {

// bf16 rows with bf16 dL/dout take the tensor-core instance.
template <int NX>
cudaError_t launch_block_bwd_nx(const BlockBwdArgs& a, cudaStream_t s) {
  const int threads = a.d / 128 * 32;
  const void* fn = a.bf16 ? (a.dz_bf16 ? reinterpret_cast<const void*>(&block_bwd_batched_kernel<bf16, bf16, NX, true>)
                                       : reinterpret_cast<const void*>(&block_bwd_batched_kernel<bf16, float, NX, false>))
                          : (a.dz_bf16 ? reinterpret_cast<const void*>(&block_bwd_batched_kernel<float, bf16, NX, false>)
                                       : reinterpret_cast<const void*>(&block_bwd_batched_kernel<float, float, NX, false>));
  const int smem = static_cast<int>(block_bwd_smem(a));
  cudaError_t e = allow_dynamic_smem(fn, smem);
  if (e != cudaSuccess) return e;
  alignas(64) CUtensorMap mv, mf;
  if (!encode_grad_maps(a, &mv, &mf)) return cudaErrorInvalidValue;
  int64_t grid = static_cast<int64_t>(sm_count()) * blocks_per_sm(fn, threads, smem);
  if (grid > a.T) grid = a.T;
  const unsigned g = static_cast<unsigned>(grid > 0 ? grid : 1);
  if (a.bf16) {
    if (a.dz_bf16) block_bwd_batched_kernel<bf16, bf16, NX, true><<<g, threads, smem, s>>>(a, mv, mf);
    else block_bwd_batched_kernel<bf16, float, NX, false><<<g, threads, smem, s>>>(a, mv, mf);
  } else {
    if (a.dz_bf16) block_bwd_batched_kernel<float, bf16, NX, false><<<g, threads, smem, s>>>(a, mv, mf);
    else block_bwd_batched_kernel<float, float, NX, false><<<g, threads, smem, s>>>(a, mv, mf);
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t take_timeout_blockbwd(unsigned int* flag) {
  unsigned int zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(flag, g_blockbwd_timeout, sizeof(unsigned int));
  if (e != cudaSuccess) return e;
  return cudaMemcpyToSymbol(g_blockbwd_timeout, &zero, sizeof(unsigned int));
}

cudaError_t launch_block_bwd_batched(const BlockBwdArgs& a, cudaStream_t s) {
  const int n1 = a.n + 1;
  return n1 <= 2 ? launch_block_bwd_nx<2>(a, s) : n1 <= 4 ? launch_block_bwd_nx<4>(a, s) : launch_block_bwd_nx<8>(a, s);
}

}  // namespace attnres
