// Projection of the input-dependent query: Q[t, :] = Wq h(t), i.e.
// Q = H Wq^T with H [T, d] and Wq [d, d] in bf16 and Q in fp32 (the ablation
// the pages report: a query projected from the current hidden state by a
// per-layer d x d matrix instead of the fixed learned pseudo-query; LLMRes
// blog, on the paper's ablation).
//
// A dense contraction, so it runs on the tensor cores: 128 x 128 output tiles
// per CTA, 8 warps of 64 x 32, K in steps of 32 staged by a 3-deep cp.async
// pipeline into shared rows padded to 80 bytes (ldmatrix without bank
// conflicts), m16n8k16 bf16 MMAs with fp32 accumulation. bf16 products are
// exact in fp32, so Q carries only the fp32 rounding of the sums.
#include "common.cuh"
#include "internal.h"

namespace attnres {
namespace {

constexpr int kPBM = 128, kPBN = 128, kPBK = 32, kPStages = 3;
constexpr int kPPitch = kPBK + 8;  // elements per staged row (80 bytes)
constexpr int kPThreads = 256;
constexpr int kPSmem = kPStages * (kPBM + kPBN) * kPPitch * 2;

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool full) {
  // src_size 0 fills the 16 bytes with zeros (rows past T).
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(full ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void ldsm_x4_p(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

__device__ __forceinline__ void mma_p(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__global__ void __launch_bounds__(kPThreads) proj_kernel(const bf16* H, const bf16* Wq, float* Q, int64_t T,
                                                         int d) {
  extern __shared__ __align__(128) unsigned char smem[];
  bf16* As = reinterpret_cast<bf16*>(smem);                         // [stages][BM][pitch]
  bf16* Bs = As + kPStages * kPBM * kPPitch;                       // [stages][BN][pitch]
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t m0 = static_cast<int64_t>(blockIdx.x) * kPBM;
  const int n0 = blockIdx.y * kPBN;
  const int wm = warp >> 2, wn = warp & 3;  // warp tile: rows wm*64.., cols wn*32..
  const int nk = d / kPBK;

  pdl_trigger();
  pdl_wait();

  // Each thread copies 2 16-byte chunks of A and 2 of B per stage.
  auto load_stage = [&](int stage, int kt) {
    const int k0 = kt * kPBK;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int c = tid + h * kPThreads;  // 0..511: row c / 4, chunk c % 4
      const int r = c >> 2, ch = c & 3;
      const int64_t row = m0 + r;
      const bool in = row < T;
      cp_async16(smem_u32(As + (stage * kPBM + r) * kPPitch + ch * 8), H + (in ? row : 0) * d + k0 + ch * 8, in);
      cp_async16(smem_u32(Bs + (stage * kPBN + r) * kPPitch + ch * 8), Wq + static_cast<int64_t>(n0 + r) * d + k0 + ch * 8,
                 true);
    }
  };

  float acc[4][4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j][0] = acc[i][j][1] = acc[i][j][2] = acc[i][j][3] = 0.f;

#pragma unroll
  for (int s = 0; s < kPStages - 1; ++s) {
    if (s < nk) load_stage(s, s);
    cp_async_commit();
  }
  const int a_row = lane & 15, a_col = (lane >> 4) * 8;
  const int b_row = (lane & 7) + ((lane >> 4) << 3), b_col = ((lane >> 3) & 1) * 8;
  for (int kt = 0; kt < nk; ++kt) {
    const int nxt = kt + kPStages - 1;
    if (nxt < nk) load_stage(nxt % kPStages, nxt);
    cp_async_commit();
    cp_async_wait<kPStages - 1>();
    __syncthreads();
    const int st = kt % kPStages;
    const bf16* Ab = As + (st * kPBM + wm * 64) * kPPitch;
    const bf16* Bb = Bs + (st * kPBN + wn * 32) * kPPitch;
#pragma unroll
    for (int kk = 0; kk < kPBK; kk += 16) {
      uint32_t af[4][4], bfr[2][4];
#pragma unroll
      for (int i = 0; i < 4; ++i) ldsm_x4_p(smem_u32(Ab + (i * 16 + a_row) * kPPitch + kk + a_col), af[i]);
#pragma unroll
      for (int j = 0; j < 2; ++j) ldsm_x4_p(smem_u32(Bb + (j * 16 + b_row) * kPPitch + kk + b_col), bfr[j]);
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) mma_p(acc[i][j], af[i], bfr[j >> 1][(j & 1) * 2], bfr[j >> 1][(j & 1) * 2 + 1]);
    }
    __syncthreads();  // the stage is overwritten by a later load
  }
  cp_async_wait<0>();

  const int g = lane >> 2, t = lane & 3;
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int col = n0 + wn * 32 + j * 8 + 2 * t;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int64_t row = m0 + wm * 64 + i * 16 + g + 8 * h;
        if (row < T)
          *reinterpret_cast<float2*>(Q + row * d + col) = make_float2(acc[i][j][2 * h], acc[i][j][2 * h + 1]);
      }
    }
}

}  // namespace

namespace {
// Any d, any alignment: one thread per output element, fp32 sums.
__global__ void __launch_bounds__(256) proj_generic_kernel(const bf16* H, const bf16* Wq, float* Q, int64_t T, int d) {
  pdl_trigger();
  pdl_wait();
  const int64_t total = T * d;
  for (int64_t e = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; e < total;
       e += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t t = e / d;
    const int j = static_cast<int>(e - t * d);
    float acc = 0.f;
    for (int k = 0; k < d; ++k) acc = fmaf(to_f32(H[t * d + k]), to_f32(Wq[static_cast<int64_t>(j) * d + k]), acc);
    Q[e] = acc;
  }
}
}  // namespace

cudaError_t launch_proj_generic(const void* H, const void* Wq, float* Q, int64_t T, int d, cudaStream_t s) {
  int64_t blocks = (T * d + 255) / 256;
  const int64_t cap = static_cast<int64_t>(sm_count()) * 8;
  if (blocks > cap) blocks = cap;
  return launch_pdl(proj_generic_kernel, static_cast<unsigned>(blocks), 256, 0, s, static_cast<const bf16*>(H),
                    static_cast<const bf16*>(Wq), Q, T, d);
}

bool proj_ok(const void* H, const void* Wq, const float* Q, int d) {
  return d % kPBN == 0 && aligned16(H) && aligned16(Wq) && aligned16(Q);
}

cudaError_t launch_proj(const void* H, const void* Wq, float* Q, int64_t T, int d, cudaStream_t s) {
  cudaError_t e = allow_dynamic_smem(reinterpret_cast<const void*>(&proj_kernel), kPSmem);
  if (e != cudaSuccess) return e;
  const int64_t mt = (T + kPBM - 1) / kPBM;
  if (mt > 0x7fffffff) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(mt), static_cast<unsigned>(d / kPBN));
  cfg.blockDim = dim3(kPThreads);
  cfg.dynamicSmemBytes = kPSmem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, proj_kernel, static_cast<const bf16*>(H), static_cast<const bf16*>(Wq), Q, T, d);
}

}  // namespace attnres
