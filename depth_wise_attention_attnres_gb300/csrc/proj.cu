// Projection of the input-dependent query: Q[t, :] = Wq h(t), i.e.
// Q = H Wq^T with H [T, d] and Wq [d, d] in bf16 and Q in fp32 (the ablation
// the pages report: a query projected from the current hidden state by a
// per-layer d x d matrix instead of the fixed learned pseudo-query; LLMRes
// blog, on the paper's ablation).
//
// A dense contraction, so it runs on the tensor cores. Four kernels, chosen
// by attnres_query_projection in this order:
//   proj_tc2_kernel, when d is a multiple of 256 and the product has at least
//     one 256 x 256 output tile for every pair of SMs the device can hold:
//     clusters of two CTAs share each tile through tcgen05.mma.cta_group::2
//     (M = 256), each CTA holding half of the tile's A rows and half of its B
//     rows (section "tcgen05 path, CTA pairs" below).
//   proj_tc_kernel, the path that runs otherwise whenever d is a multiple of
//     128, 160, 192, 224 or 256, the operands are 16-byte aligned and the
//     driver can encode tensor maps: 5th-generation tensor cores. Persistent,
//     one CTA per SM over 128 x BN output tiles; a TMA warp streams
//     128-byte-swizzled operand stages, one thread issues tcgen05.mma
//     (M = 128, N = BN, K = 16) into one of two fp32 accumulators in tensor
//     memory, and four epilogue warps drain the other with tcgen05.ld through
//     a small shared staging block (section "tcgen05 path" below).
//   proj_kernel (fallback when no tensor map is available, d a multiple of
//     128): warp-level m16n8k16 bf16 MMAs, 128 x 128 tiles per CTA, 8 warps of
//     64 x 32, K in steps of 32 staged by a 3-deep cp.async pipeline into
//     rows padded to 80 bytes (ldmatrix without bank conflicts).
//   proj_generic_kernel: any other shape, plain fp32 FMAs.
// bf16 products are exact in fp32, so Q carries only the fp32 rounding of
// the sums on every path.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>
#include <utility>
#include <vector>

#include "common.cuh"
#include "internal.h"

namespace attnres {
namespace {

constexpr int kPBM = 128, kPBN = 128, kPBK = 32, kPStages = 3;
constexpr int kPPitch = kPBK + 8;  // elements per staged row (80 bytes)
constexpr int kPThreads = 256;
constexpr int kPSmem = kPStages * (kPBM + kPBN) * kPPitch * 2;


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
      for (int i = 0; i < 4; ++i) ldsm_x4(smem_u32(Ab + (i * 16 + a_row) * kPPitch + kk + a_col), af[i]);
#pragma unroll
      for (int j = 0; j < 2; ++j) ldsm_x4(smem_u32(Bb + (j * 16 + b_row) * kPPitch + kk + b_col), bfr[j]);
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) mma16816(acc[i][j], af[i], bfr[j >> 1][(j & 1) * 2], bfr[j >> 1][(j & 1) * 2 + 1]);
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


// ------------------------------------------------------------ tcgen05 path --
// The same GEMM on the 5th-generation tensor cores: 128 x BN output tiles,
// the fp32 accumulator in tensor memory (128 lanes x BN columns). Operand
// tiles of 128 (A) and BN (B) rows x 64 K (one 128-byte swizzle atom per row)
// arrive by 2-d TMA copies with the 128-byte swizzle into 4 stages; one thread
// issues tcgen05.mma (M = 128, N = BN, K = 16, bf16 x bf16 -> fp32), and
// tcgen05.commit frees a stage once the MMAs that read it are done. The four
// epilogue warps then read their 32-lane quarter of the accumulator with
// tcgen05.ld and store it through a small shared-memory staging block, as
// whole 128-byte row segments. Every wait is bounded; whatever happens, the CTA waits for
// the MMAs it issued and the copies in flight and frees its tensor memory.
namespace {

__device__ unsigned int g_proj_timeout = 0;

// Output tiles of 128 rows x BN columns (BN up to 256, the widest tcgen05
// N; wider tiles read fewer operand bytes per product from L2).
constexpr int kTBM = 128, kTBK = 64, kTStages = 4;
constexpr int kTTileBytes = kTBM * kTBK * 2;           // the A tile of a stage, 16 KB
// Epilogue staging: per epilogue warp, a 32 x 32 fp32 block in rows of 36
// floats (16-byte aligned; 16-byte accesses by 8 lanes hit distinct banks).
constexpr int kEpiLd = 36, kEpiWarpFloats = 32 * kEpiLd;
template <int BN> struct TcTile {
  static constexpr int kStageBytes = kTTileBytes + BN * kTBK * 2;  // A and B
  static constexpr int kSmem = 1024 + kTStages * kStageBytes + 128 + 4 * kEpiWarpFloats * 4;
  static constexpr uint32_t kTmemCols = BN <= 128 ? 128u : 256u;     // a power of two >= BN
  // Instruction descriptor of tcgen05.mma kind::f16: fp32 accumulator (bits
  // 4-5), bf16 A (7-9) and B (10-12), both K-major (15, 16), N / 8 (17-22),
  // M / 16 (24-28).
  static constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(BN >> 3) << 17) |
                                     (static_cast<uint32_t>(kTBM >> 4) << 24);
};

// Shared-memory descriptor of a K-major operand tile in the 128-byte swizzle
// (8-row atoms of 128-byte rows, 1024 bytes apart): start address / 16 (bits
// 0-13), leading offset (ignored for this layout, 1), stride offset 1024 / 16
// (32-45), descriptor version 1 (46-47), layout SWIZZLE_128B = 2 (61-63).
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  return static_cast<uint64_t>((saddr >> 4) & 0x3FFFu) | (static_cast<uint64_t>(1) << 16) |
         (static_cast<uint64_t>(1024 >> 4) << 32) | (static_cast<uint64_t>(1) << 46) |
         (static_cast<uint64_t>(2) << 61);
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
      ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void umma_bf16(uint32_t tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}"
      ::"r"(tmem), "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void umma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// Persistent: one CTA per SM walks its share of the output tiles (tile
// blockIdx.x + i * gridDim.x; the BN-wide column tiles of one row block are
// adjacent, so CTAs running at the same time share their A rows in L2).
// Roles: warp 0 lane 0 streams operand stages by TMA; warp 1 owns the tensor
// memory and its lane 0 issues the MMAs; warps 2-5 drain accumulators. Two
// accumulators in tensor memory take turns, so a tile's epilogue runs while
// the next tile's MMAs fill the other one.
constexpr int kTcWarps = 6;
constexpr int kTcThreads = kTcWarps * 32;

template <int BN>
__global__ void __launch_bounds__(kTcThreads, 1)
    proj_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, float* Q,
                   int64_t T, int d) {
  using G = TcTile<BN>;
  constexpr int kTStageBytes = G::kStageBytes;
  constexpr uint32_t kAccCols = G::kTmemCols;  // one accumulator
  constexpr uint32_t kCols = 2 * kAccCols;     // two (a power of two, at most 512)
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem + kTStages * kTStageBytes);
  uint64_t* empty_bar = full_bar + kTStages;
  uint64_t* tfull = empty_bar + kTStages;   // [2] accumulator ready
  uint64_t* tempty = tfull + 2;             // [2] accumulator drained
  uint64_t* done_bar = tempty + 2;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(done_bar + 1);
  float* epi_stage = reinterpret_cast<float*>(smem + kTStages * kTStageBytes + 128);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ntn = d / BN;
  const int64_t ntiles = ((T + kTBM - 1) / kTBM) * ntn;
  const int nk = d / kTBK;
  const int64_t mine = blockIdx.x < ntiles ? (ntiles - 1 - blockIdx.x) / gridDim.x + 1 : 0;

  pdl_trigger();
  if (warp == 0 && lane == 0) {
    for (int s = 0; s < kTStages; ++s) {
      mbar_init(smem_u32(&full_bar[s]), 1);
      mbar_init(smem_u32(&empty_bar[s]), 1);
    }
    for (int k = 0; k < 2; ++k) {
      mbar_init(smem_u32(&tfull[k]), 1);
      mbar_init(smem_u32(&tempty[k]), 4);  // one arrival per epilogue warp
    }
    mbar_init(smem_u32(done_bar), 1);
    mbar_fence_init();
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_holder)),
                 "r"(kCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = *tmem_holder;
  pdl_wait();

  bool ok = true;
  if (warp == 0) {
    if (lane == 0) {
      // Producer: per tile, nk stages of A rows m0.. and B rows n0.., 64 K each.
      int s = 0;
      uint32_t phase = 0;
      int64_t issued = 0;
      for (int64_t i = 0; i < mine && ok; ++i) {
        const int64_t tile = blockIdx.x + i * gridDim.x;
        const int m0 = static_cast<int>(tile / ntn) * kTBM, n0 = static_cast<int>(tile % ntn) * BN;
        for (int kt = 0; kt < nk; ++kt) {
          if (!mbar_wait(smem_u32(&empty_bar[s]), phase ^ 1u)) {
            ok = false;
            break;
          }
          const uint32_t fb = smem_u32(&full_bar[s]);
          mbar_arrive_expect_tx(fb, kTStageBytes);
          const uint32_t st = smem_u32(smem + s * kTStageBytes);
          tma_load_2d(st, &tmA, kt * kTBK, m0, fb);
          tma_load_2d(st + kTTileBytes, &tmB, kt * kTBK, n0, fb);
          ++issued;
          if (++s == kTStages) {
            s = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {
        atomicOr(&g_proj_timeout, 1u);
        for (int64_t it = issued > kTStages ? issued - kTStages : 0; it < issued; ++it)
          (void)mbar_wait(smem_u32(&full_bar[it % kTStages]), static_cast<uint32_t>((it / kTStages) & 1));
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      // MMA issuer: accumulator i & 1 for the i-th tile, once drained.
      int s = 0;
      uint32_t phase = 0;
      for (int64_t i = 0; i < mine && ok; ++i) {
        const int acc = static_cast<int>(i & 1);
        if (!mbar_wait(smem_u32(&tempty[acc]), static_cast<uint32_t>(((i >> 1) & 1) ^ 1))) {
          ok = false;
          break;
        }
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        const uint32_t tacc = tmem + static_cast<uint32_t>(acc) * kAccCols;
        for (int kt = 0; kt < nk; ++kt) {
          if (!mbar_wait(smem_u32(&full_bar[s]), phase)) {
            ok = false;
            break;
          }
          asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
          const uint32_t st = smem_u32(smem + s * kTStageBytes);
          const uint64_t da = sw128_desc(st), db = sw128_desc(st + kTTileBytes);
#pragma unroll
          for (int k = 0; k < kTBK / 16; ++k)
            umma_bf16(tacc, da + static_cast<uint64_t>(k * 2), db + static_cast<uint64_t>(k * 2), G::kIdesc,
                      (kt | k) != 0);
          umma_commit(smem_u32(&empty_bar[s]));
          if (++s == kTStages) {
            s = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit(smem_u32(&tfull[acc]));
      }
      if (!ok) atomicOr(&g_proj_timeout, 1u);
      // Signals once every MMA issued above is done (also after a timeout).
      umma_commit(smem_u32(done_bar));
    }
    __syncwarp();
  } else {
    // Epilogue: warp w reads tensor-memory lanes 32 (w % 4) .. of the tile
    // (lane = row), 32 columns at a time, and turns each 32 x 32 block
    // around in shared memory so one store instruction writes four whole
    // 128-byte row segments.
    const int q4 = warp & 3;
    float* stg = epi_stage + (warp - 2) * kEpiWarpFloats;
    for (int64_t i = 0; i < mine; ++i) {
      const int acc = static_cast<int>(i & 1);
      const bool got = __all_sync(0xffffffffu, mbar_wait(smem_u32(&tfull[acc]), static_cast<uint32_t>((i >> 1) & 1)));
      if (!got) {
        ok = false;
        break;
      }
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      const int64_t tile = blockIdx.x + i * gridDim.x;
      const int64_t rbase = (tile / ntn) * kTBM + q4 * 32;
      const int n0 = static_cast<int>(tile % ntn) * BN;
      const uint32_t taddr = tmem + (static_cast<uint32_t>(q4 * 32) << 16) + static_cast<uint32_t>(acc) * kAccCols;
#pragma unroll 1
      for (int c = 0; c < BN / 32; ++c) {
        float v[32];
        tmem_ld32(taddr + static_cast<uint32_t>(c * 32), v);
#pragma unroll
        for (int e = 0; e < 8; ++e)
          *reinterpret_cast<float4*>(stg + lane * kEpiLd + 4 * e) =
              make_float4(v[4 * e], v[4 * e + 1], v[4 * e + 2], v[4 * e + 3]);
        __syncwarp();
#pragma unroll
        for (int h = 0; h < 8; ++h) {
          const int r = h * 4 + (lane >> 3);
          const float4 x = *reinterpret_cast<const float4*>(stg + r * kEpiLd + 4 * (lane & 7));
          if (rbase + r < T)
            *reinterpret_cast<float4*>(Q + (rbase + r) * d + n0 + c * 32 + 4 * (lane & 7)) = x;
        }
        __syncwarp();
      }
      asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&tempty[acc]));
    }
    if (!ok && lane == 0) atomicOr(&g_proj_timeout, 1u);
  }
  // Teardown: every issued MMA has finished before the tensor memory goes.
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (warp == 1) {
    if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(done_bar), 0)) && lane == 0) atomicOr(&g_proj_timeout, 1u);
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kCols) : "memory");
  }
}

// ------------------------------------------------ tcgen05 path, CTA pairs --
// Clusters of two CTAs on two SMs share each 256 x BN output tile through
// tcgen05.mma.cta_group::2 (M = 256). CTA r of a pair holds rows
// 128 r .. 128 r + 127 of the tile's A block and rows r BN/2 .. r BN/2 +
// BN/2 - 1 of its B block (output columns); the MMAs, issued by one thread of
// the even CTA, read both CTAs' shared memory and leave each CTA's 128 rows of
// the accumulator in that CTA's own tensor memory. Per K step an SM so takes
// in 128 + BN/2 operand rows for its 128 x BN share of the product, where a
// CTA alone takes in 128 + BN.
//
// Barriers (every wait bounded):
//  * full[s], in the even CTA: its producer arms the phase with the bytes of
//    both CTAs' copies, and the copies of both producers (the cta_group::2
//    form of the TMA load, which may signal the peer's barrier) complete on it;
//  * empty[s] and tfull[a], in both CTAs: the MMA thread's commits arrive on
//    the barrier at the same offset in both CTAs (multicast);
//  * tempty[a], in the even CTA: each epilogue warp of both CTAs arrives after
//    reading its share of accumulator a;
//  * done, in both CTAs: a last multicast commit once every MMA has finished.
// Teardown: each CTA waits for done, the pair meets at a cluster barrier (so
// no CTA leaves while its peer may still touch its shared memory), and both
// free the tensor memory together.
constexpr int kT2Epi = 8;  // epilogue warps per CTA: two per tensor-memory lane quarter
constexpr int kT2Warps = 2 + kT2Epi;
constexpr int kT2Threads = kT2Warps * 32;
constexpr int kT2SmemMax = 227 * 1024;
constexpr int kT2Fixed = 1024 + 256 + kT2Epi * kEpiWarpFloats * 4;  // alignment slack, barriers, staging
template <int BN> struct Tc2Tile {
  static constexpr int kBRows = BN / 2;  // B rows a CTA holds
  static constexpr int kStageBytes = kTTileBytes + kBRows * kTBK * 2;
  static constexpr int kStages = (kT2SmemMax - kT2Fixed) / kStageBytes < 8 ? (kT2SmemMax - kT2Fixed) / kStageBytes : 8;
  static constexpr int kSmem = kT2Fixed + kStages * kStageBytes;
  static constexpr uint32_t kTmemCols = BN <= 128 ? 128u : 256u;
  // As TcTile's descriptor, with M = 256.
  static constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(BN >> 3) << 17) |
                                     (static_cast<uint32_t>(256 >> 4) << 24);
  static_assert(kBRows % 8 == 0, "B rows come in 8-row swizzle atoms");
  static_assert(kStages >= 4, "at least four operand stages");
};

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// The shared::cluster address of the same shared-memory offset in CTA `rank`.
__device__ __forceinline__ uint32_t cluster_addr(uint32_t local, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
  return r;
}

// All threads of both CTAs; orders each thread's earlier memory operations
// (remote arrivals included) before the other CTA's later ones.
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_remote(uint32_t caddr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(caddr) : "memory");
}

// mbar_wait for barriers that other CTAs of the cluster signal.
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n"
      " mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ bool mbar_wait_cluster(uint32_t bar, uint32_t parity) {
  if (mbar_try_wait_cluster(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 32; ++i)
      if (mbar_try_wait_cluster(bar, parity)) return true;
    if (global_ns() - t0 > kWaitLimitNs) return false;
  }
}

// TMA tile load whose completion may be signalled on the peer CTA's barrier
// (`bar` a shared::cluster address).
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
      "[%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void umma_bf16_pair(uint32_t tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                               uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrives once on the barrier at offset `bar` in both CTAs of the pair when
// the MMAs issued so far have finished.
__device__ __forceinline__ void umma_commit_pair(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(bar),
      "h"(static_cast<uint16_t>(3))
      : "memory");
}

// Persistent over pair tiles: pair p = blockIdx.x / 2 takes tiles
// p + i * (gridDim.x / 2). Roles in each CTA: warp 0 lane 0 streams this
// CTA's operand rows by TMA; warp 1 holds the tensor memory (both CTAs take
// part in its allocation) and, in the even CTA, its lane 0 issues the MMAs;
// warps 2-9 drain the accumulators, two warps per lane quarter, splitting
// the 32-column blocks between them.
template <int BN>
__global__ void __launch_bounds__(kT2Threads, 1)
    proj_tc2_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, float* Q,
                    int64_t T, int d) {
  using G = Tc2Tile<BN>;
  constexpr int kS = G::kStages;
  constexpr uint32_t kAccCols = G::kTmemCols;
  constexpr uint32_t kCols = 2 * kAccCols;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem + kS * G::kStageBytes);
  uint64_t* empty_bar = full_bar + kS;
  uint64_t* tfull = empty_bar + kS;   // [2]
  uint64_t* tempty = tfull + 2;       // [2]
  uint64_t* done_bar = tempty + 2;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(done_bar + 1);
  float* epi_stage = reinterpret_cast<float*>(smem + kS * G::kStageBytes + 256);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  const int64_t pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;
  const int ntn = d / BN;
  const int64_t ntiles = ((T + 255) / 256) * ntn;
  const int nk = d / kTBK;
  const int64_t mine = pair < ntiles ? (ntiles - 1 - pair) / npairs + 1 : 0;

  pdl_trigger();
  if (warp == 0 && lane == 0) {
    for (int s = 0; s < kS; ++s) {
      mbar_init(smem_u32(&full_bar[s]), 1);
      mbar_init(smem_u32(&empty_bar[s]), 1);
    }
    for (int k = 0; k < 2; ++k) {
      mbar_init(smem_u32(&tfull[k]), 1);
      mbar_init(smem_u32(&tempty[k]), 2 * kT2Epi);
    }
    mbar_init(smem_u32(done_bar), 1);
    mbar_fence_init();
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_holder)),
                 "r"(kCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  cluster_sync();  // both CTAs' barriers are initialised before any remote use
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = *tmem_holder;
  pdl_wait();

  bool ok = true;
  if (warp == 0) {
    if (lane == 0) {
      int s = 0;
      uint32_t phase = 0;
      int64_t issued = 0;
      for (int64_t i = 0; i < mine && ok; ++i) {
        const int64_t tile = pair + i * npairs;
        const int m0 = static_cast<int>(tile / ntn) * 256 + static_cast<int>(rank) * kTBM;
        const int n0 = static_cast<int>(tile % ntn) * BN + static_cast<int>(rank) * G::kBRows;
        for (int kt = 0; kt < nk; ++kt) {
          if (!mbar_wait(smem_u32(&empty_bar[s]), phase ^ 1u)) {
            ok = false;
            break;
          }
          const uint32_t fb = smem_u32(&full_bar[s]);
          if (rank == 0) mbar_arrive_expect_tx(fb, 2 * G::kStageBytes);
          const uint32_t fbc = cluster_addr(fb, 0);
          const uint32_t st = smem_u32(smem + s * G::kStageBytes);
          tma_load_2d_pair(st, &tmA, kt * kTBK, m0, fbc);
          tma_load_2d_pair(st + kTTileBytes, &tmB, kt * kTBK, n0, fbc);
          ++issued;
          if (++s == kS) {
            s = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {
        atomicOr(&g_proj_timeout, 1u);
        // The even CTA's full barriers count both CTAs' copies; once the
        // phases it armed complete, no copy of either CTA is in flight.
        if (rank == 0)
          for (int64_t it = issued > kS ? issued - kS : 0; it < issued; ++it)
            (void)mbar_wait_cluster(smem_u32(&full_bar[it % kS]), static_cast<uint32_t>((it / kS) & 1));
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (rank == 0 && lane == 0) {
      int s = 0;
      uint32_t phase = 0;
      for (int64_t i = 0; i < mine && ok; ++i) {
        const int acc = static_cast<int>(i & 1);
        if (!mbar_wait_cluster(smem_u32(&tempty[acc]), static_cast<uint32_t>(((i >> 1) & 1) ^ 1))) {
          ok = false;
          break;
        }
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        const uint32_t tacc = tmem + static_cast<uint32_t>(acc) * kAccCols;
        for (int kt = 0; kt < nk; ++kt) {
          if (!mbar_wait_cluster(smem_u32(&full_bar[s]), phase)) {
            ok = false;
            break;
          }
          asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
          const uint32_t st = smem_u32(smem + s * G::kStageBytes);
          const uint64_t da = sw128_desc(st), db = sw128_desc(st + kTTileBytes);
#pragma unroll
          for (int k = 0; k < kTBK / 16; ++k)
            umma_bf16_pair(tacc, da + static_cast<uint64_t>(k * 2), db + static_cast<uint64_t>(k * 2), G::kIdesc,
                           (kt | k) != 0);
          umma_commit_pair(smem_u32(&empty_bar[s]));
          if (++s == kS) {
            s = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit_pair(smem_u32(&tfull[acc]));
      }
      if (!ok) atomicOr(&g_proj_timeout, 1u);
      umma_commit_pair(smem_u32(done_bar));
    }
    __syncwarp();
  } else {
    const int q4 = warp & 3;
    const int half = (warp - 2) >> 2;
    float* stg = epi_stage + (warp - 2) * kEpiWarpFloats;
    const uint32_t tempty_c0 = cluster_addr(smem_u32(&tempty[0]), 0);
    const uint32_t tempty_c1 = cluster_addr(smem_u32(&tempty[1]), 0);
    for (int64_t i = 0; i < mine; ++i) {
      const int acc = static_cast<int>(i & 1);
      const bool got =
          __all_sync(0xffffffffu, mbar_wait_cluster(smem_u32(&tfull[acc]), static_cast<uint32_t>((i >> 1) & 1)));
      if (!got) {
        ok = false;
        break;
      }
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      const int64_t tile = pair + i * npairs;
      const int64_t rbase = (tile / ntn) * 256 + static_cast<int64_t>(rank) * kTBM + q4 * 32;
      const int n0 = static_cast<int>(tile % ntn) * BN;
      const uint32_t taddr = tmem + (static_cast<uint32_t>(q4 * 32) << 16) + static_cast<uint32_t>(acc) * kAccCols;
#pragma unroll 1
      for (int c = half; c < BN / 32; c += 2) {
        float v[32];
        tmem_ld32(taddr + static_cast<uint32_t>(c * 32), v);
#pragma unroll
        for (int e = 0; e < 8; ++e)
          *reinterpret_cast<float4*>(stg + lane * kEpiLd + 4 * e) =
              make_float4(v[4 * e], v[4 * e + 1], v[4 * e + 2], v[4 * e + 3]);
        __syncwarp();
#pragma unroll
        for (int h = 0; h < 8; ++h) {
          const int r = h * 4 + (lane >> 3);
          const float4 x = *reinterpret_cast<const float4*>(stg + r * kEpiLd + 4 * (lane & 7));
          if (rbase + r < T)
            *reinterpret_cast<float4*>(Q + (rbase + r) * d + n0 + c * 32 + 4 * (lane & 7)) = x;
        }
        __syncwarp();
      }
      asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
      __syncwarp();
      if (lane == 0) mbar_arrive_remote(acc ? tempty_c1 : tempty_c0);
    }
    if (!ok && lane == 0) atomicOr(&g_proj_timeout, 1u);
  }
  // Teardown: every MMA has finished (done), then neither CTA leaves or frees
  // the tensor memory before the other is through.
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (warp == 1 && !__all_sync(0xffffffffu, mbar_wait_cluster(smem_u32(done_bar), 0)) && lane == 0)
    atomicOr(&g_proj_timeout, 1u);
  cluster_sync();
  if (warp == 1) {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kCols) : "memory");
  }
}

// A [rows, d] bf16 operand as a 2-d tensor, box {64, box_rows}, 128-byte swizzle.
bool encode_operand(const void* base, int64_t rows, int d, int box_rows, CUtensorMap* map) {
  PFN_cuTensorMapEncodeTiled_v12000 fn = tensor_map_encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(d) * 2};
  const cuuint32_t box[2] = {kTBK, static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t es[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Output tile width: the widest that divides d (fewer operand bytes per
// product), except when 128-wide tiles fit in one wave over the SMs, where
// more tiles spread the work further. At 8192 x 896 the widest (224) takes
// 14.4 us against 16.8 us for 128-wide tiles.
inline int proj_tile_n(int d, int64_t T) {
  if (d % 128 == 0 && ((T + kTBM - 1) / kTBM) * (d / 128) <= static_cast<int64_t>(sm_count())) return 128;
  const int cands[5] = {256, 224, 192, 160, 128};
  for (int c : cands)
    if (d % c == 0) return c;
  return 0;
}

template <int BN>
cudaError_t launch_proj_tc_n(const void* H, const void* Wq, float* Q, int64_t T, int d, cudaStream_t s) {
  alignas(64) CUtensorMap ma, mb;
  if (!encode_operand(H, T, d, kTBM, &ma) || !encode_operand(Wq, d, d, BN, &mb)) return cudaErrorInvalidValue;
  constexpr int kTSmem = TcTile<BN>::kSmem;
  cudaError_t e = allow_dynamic_smem(reinterpret_cast<const void*>(&proj_tc_kernel<BN>), kTSmem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  const int64_t tiles = ((T + kTBM - 1) / kTBM) * (d / BN);
  int64_t grid = sm_count();
  if (grid > tiles) grid = tiles;
  cfg.gridDim = dim3(static_cast<unsigned>(grid > 0 ? grid : 1));
  cfg.blockDim = dim3(kTcThreads);
  cfg.dynamicSmemBytes = kTSmem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, proj_tc_kernel<BN>, ma, mb, Q, T, d);
}

cudaError_t launch_proj_tc(const void* H, const void* Wq, float* Q, int64_t T, int d, cudaStream_t s) {
  switch (proj_tile_n(d, T)) {
    case 256: return launch_proj_tc_n<256>(H, Wq, Q, T, d, s);
    case 224: return launch_proj_tc_n<224>(H, Wq, Q, T, d, s);
    case 192: return launch_proj_tc_n<192>(H, Wq, Q, T, d, s);
    case 160: return launch_proj_tc_n<160>(H, Wq, Q, T, d, s);
    case 128: return launch_proj_tc_n<128>(H, Wq, Q, T, d, s);
    default: return cudaErrorInvalidValue;
  }
}

// Launch configuration of the pair kernel with its cluster attribute.
template <int BN>
void pair_config(cudaLaunchConfig_t& cfg, cudaLaunchAttribute (&attr)[2], int64_t pairs, cudaStream_t s) {
  cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(2 * pairs));
  cfg.blockDim = dim3(kT2Threads);
  cfg.dynamicSmemBytes = Tc2Tile<BN>::kSmem;
  cfg.stream = s;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
}

// How many CTA pairs of the pair kernel fit on the device at once (0 when
// clusters cannot be launched), asked once per device and tile width.
template <int BN>
int pair_slots() {
  static std::mutex mu;
  static std::vector<std::pair<int, int>> known;  // (device, pairs)
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  std::lock_guard<std::mutex> lk(mu);
  for (const auto& k : known)
    if (k.first == dev) return k.second;
  int n = 0;
  if (allow_dynamic_smem(reinterpret_cast<const void*>(&proj_tc2_kernel<BN>), Tc2Tile<BN>::kSmem) == cudaSuccess) {
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attr[2];
    pair_config<BN>(cfg, attr, sm_count() / 2, nullptr);
    cfg.numAttrs = 1;  // the occupancy query takes the cluster shape only
    if (cudaOccupancyMaxActiveClusters(&n, proj_tc2_kernel<BN>, &cfg) != cudaSuccess) n = 0;
  }
  (void)cudaGetLastError();
  known.emplace_back(dev, n);
  return n;
}

// Pair tile width for the pair kernel, 0 when it does not serve the shape.
// Pairs pay with 256-wide tiles: measured at 16384 x 1024 and 8192 x 2048,
// 30.3 and 47.4 us against 33.4 and 52.3 us for single CTAs. With 224-wide
// tiles (d = 896) they tie with single CTAs (14.6 against 14.1 us at 8192
// rows) and with 128-wide ones they lose (17.1 us): there an SM's K steps
// are set by the MMAs and the operand copies together, not by the operand
// bytes. The 256-row tiles must also give every pair slot a tile.
inline int proj2_tile_n(int d, int64_t T) {
  if (d % 256 != 0) return 0;
  const int slots = pair_slots<256>();
  return slots >= 1 && ((T + 255) / 256) * (d / 256) >= slots ? 256 : 0;
}

template <int BN>
cudaError_t launch_proj_tc2_n(const void* H, const void* Wq, float* Q, int64_t T, int d, cudaStream_t s) {
  alignas(64) CUtensorMap ma, mb;
  if (!encode_operand(H, T, d, kTBM, &ma) || !encode_operand(Wq, d, d, BN / 2, &mb)) return cudaErrorInvalidValue;
  cudaError_t e = allow_dynamic_smem(reinterpret_cast<const void*>(&proj_tc2_kernel<BN>), Tc2Tile<BN>::kSmem);
  if (e != cudaSuccess) return e;
  const int64_t tiles = ((T + 255) / 256) * (d / BN);
  int64_t pairs = pair_slots<BN>();
  if (pairs > tiles) pairs = tiles;
  if (pairs < 1) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg;
  cudaLaunchAttribute attr[2];
  pair_config<BN>(cfg, attr, pairs, s);
  return cudaLaunchKernelEx(&cfg, proj_tc2_kernel<BN>, ma, mb, Q, T, d);
}

}  // namespace

bool proj_tc_ok(const void* H, const void* Wq, const float* Q, int64_t T, int d) {
  return proj_tile_n(d, T) != 0 && aligned16(H) && aligned16(Wq) && aligned16(Q) && T < (int64_t(1) << 31) &&
         (T + kTBM - 1) / kTBM <= 0x7fffffff && tensor_map_encode_fn() != nullptr;
}

cudaError_t take_timeout_proj(unsigned int* flag) {
  unsigned int zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(flag, g_proj_timeout, sizeof(unsigned int));
  if (e != cudaSuccess) return e;
  return cudaMemcpyToSymbol(g_proj_timeout, &zero, sizeof(unsigned int));
}

cudaError_t launch_proj_tensor(const void* H, const void* Wq, float* Q, int64_t T, int d, cudaStream_t s) {
  return proj2_tile_n(d, T) ? launch_proj_tc2_n<256>(H, Wq, Q, T, d, s) : launch_proj_tc(H, Wq, Q, T, d, s);
}

int proj_path(const void* H, const void* Wq, const float* Q, int64_t T, int d) {
  if (proj_tc_ok(H, Wq, Q, T, d)) return proj2_tile_n(d, T) ? 2 : 1;
  return 0;
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
