// Block stage 1 split over the feature dimension (datacamp explainer, system
// optimisations, "memory-efficient prefill": the block representations are
// sharded across tensor-parallel devices for 128K+ contexts). Read here as a
// split of the features: each device keeps a slice of every source row, and
// only the score statistics are exchanged.
//
// A shard holds features [k0, k0 + d_s) of every source row. For the read of
// query j over source i at token t the score needs
//   ss_it = sum_k v_itk^2   and   dot_ijt = sum_k w_jk gamma_jk v_itk
// over all d features; they are sums, so each shard forms its part and the
// parts are added (the one exchange step: an all-reduce of (1 + S) floats per
// (source, token)). Here the shards of one GPU add into one buffer in turn.
// With the totals each shard computes the scores e_ijt = dot_ijt /
// sqrt(ss_it / d + eps), the softmax over sources, lse, and the weighted sums
// of its own features.
//
// Partials are stored token-major, partials[t][i][c] (c = 0: sum v^2, 1 + j:
// dot_j), so one token's statistics are contiguous.
// dsplit_partials_tc_kernel (bf16, shard width a multiple of 64): the sources
// streamed by TMA into a ring shared by up to 15 consumer warps behind one
// producer warp, the dots and sum v^2 as tensor-core MMAs over 16-pair tiles.
// dsplit_partials_kernel (the rest): 8 lanes per (token, source) row of the
// shard (4 rows per warp), w * gamma of the shard in shared memory, sums over
// the row's lanes with 3 shuffle steps.
// Both write (or add to) the partials.
// dsplit_finish_kernel: one warp per token; lanes take the scores of (source,
// query) pairs from the token's partials, one lane per query takes the
// softmax, then each lane reads its features of each source once (loads one
// batch ahead of the math) and forms all S weighted sums, and stores the
// shard's output slices.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <math.h>

#include "common.cuh"
#include "internal.h"

namespace attnres {
namespace {

constexpr int kDWarps = 8;
constexpr int kDsplitSmemLimit = 227 * 1024;
constexpr int kPartMaxWarps = 15;  // consumer warps of the partials (16 warps: 128 registers each)

// bf16 elements per row of the w * gamma tables of the tensor-core partials:
// a row pitch of 64 mod 128 bytes, so the two rows one 8-lane phase of a
// 16-byte shared load reads fall in different banks.
__host__ __device__ inline int tc_pitch(int ds) { return (((ds * 2 + 127) / 128) * 128 + 64) / 2; }

inline int finish_smem(const DsplitArgs& a) { return kDWarps * a.n_src * ((a.S + 3) & ~3) * 4; }

template <typename T>
__global__ void __launch_bounds__(kDWarps * 32) dsplit_partials_kernel(DsplitArgs a) {
  extern __shared__ float wq[];  // [S][d_s] w * gamma of the shard
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int S = a.S, ds = a.d_shard, n = a.n_src;
  const int sub = lane >> 3, sl = lane & 7;  // 4 rows per warp, 8 lanes per row
  pdl_trigger();
  pdl_wait();
  for (int i = threadIdx.x; i < S * ds; i += blockDim.x) wq[i] = a.W[i] * a.Gamma[i];
  __syncthreads();
  const int64_t rows = static_cast<int64_t>(n) * a.T;
  for (int64_t r0 = (static_cast<int64_t>(blockIdx.x) * kDWarps + warp) * 4; r0 < rows;
       r0 += static_cast<int64_t>(gridDim.x) * kDWarps * 4) {
    const int64_t r = r0 + sub;  // row = token-major (t, i): its partials are contiguous
    const bool live = r < rows;
    const int64_t t = live ? r / n : 0;
    const int i = live ? static_cast<int>(r - t * n) : 0;
    const T* v = static_cast<const T*>(a.Src) + i * a.src_stride + t * ds;
    float ss = 0.f, dot[ATTNRES_MAX_QUERIES];
#pragma unroll
    for (int j = 0; j < ATTNRES_MAX_QUERIES; ++j) dot[j] = 0.f;
    if (live) {
      for (int k = sl * 4; k < ds; k += 8 * 4) {
        float x[4];
        ldg4(v + k, x);
        ss = fmaf(x[0], x[0], fmaf(x[1], x[1], fmaf(x[2], x[2], fmaf(x[3], x[3], ss))));
#pragma unroll
        for (int j = 0; j < ATTNRES_MAX_QUERIES; ++j)
          if (j < S) {
            const float4 w4 = *reinterpret_cast<const float4*>(wq + j * ds + k);
            dot[j] = fmaf(w4.x, x[0], fmaf(w4.y, x[1], fmaf(w4.z, x[2], fmaf(w4.w, x[3], dot[j]))));
          }
      }
    }
    // Sums over the 8 lanes of the row.
#pragma unroll
    for (int off = 1; off < 8; off <<= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
#pragma unroll
    for (int j = 0; j < ATTNRES_MAX_QUERIES; ++j)
      if (j < S) {
#pragma unroll
        for (int off = 1; off < 8; off <<= 1) dot[j] += __shfl_xor_sync(0xffffffffu, dot[j], off);
      }
    if (live) {
      float* pr = a.partials + r * (S + 1);
      // Lane sl of the row writes entries sl, sl + 8 (contiguous stores).
      for (int c = sl; c < S + 1; c += 8) {
        float val = ss;
#pragma unroll
        for (int j = 0; j < ATTNRES_MAX_QUERIES; ++j)
          if (c == 1 + j) val = dot[j];
        pr[c] = a.accumulate ? pr[c] + val : val;
      }
    }
  }
}

// bf16 shards whose width is a multiple of 64: the dots on the tensor cores,
// the sources streamed by TMA. A stage holds the box {64 features, n
// sources, TM tokens, d_s / 64 chunks} of TM tokens
// (TM * n = P (token, source) pairs, about 16), stored with the 128-byte
// swizzle: pair p's features of chunk c form 128-byte line L = c * P + p, and
// its 16-byte unit u lies at unit u ^ (L & 7) of the line.
// The warp takes 16 pairs at a time as the A operand of m16n8k16 MMAs and
// w * gamma (split into bf16 hi + lo, so the product keeps about 16 mantissa
// bits) as B, 8 queries per N tile. Lane (g, q) reads 16 contiguous bytes of
// its two pairs per 32 features straight into A fragments: the dot is a sum,
// so the order of k inside a lane quad's 32 features is free, as long as B's
// fragments take the same order. MMA row g holds pair sigma(g) = 4 (g & 1) +
// g / 2, so the two rows one 8-lane phase of a 16-byte shared load reads are
// 4 lines apart and their units fall in different banks. sum v^2 is the
// diagonal of A A^T, on the tensor cores too.
struct PtGeom {
  int TM, P, mtiles;    // tokens per box, pairs per box, 16-pair MMA tiles per box
  int W, nst;           // warps per CTA, stages per warp
  int box_bytes, stage_bytes;
  int tab_off, bar_off, total;
};

// Ring geometry: tab_fixed bytes shared by the CTA plus tab_warp bytes per
// warp after the rings; the most bytes in flight that fit.
inline PtGeom ring_geom(int n, int ds, int tab_fixed, int tab_warp) {
  PtGeom g{};
  g.TM = n <= 16 ? 16 / n : 1;
  g.P = g.TM * n;
  g.mtiles = (g.P + 15) / 16;
  g.box_bytes = g.P * ds * 2;
  g.stage_bytes = (g.box_bytes + 1023) / 1024 * 1024;
  int64_t best = -1;
  const int ws[4] = {8, 4, 2, 1};
  for (int wi = 0; wi < 4; ++wi)
    for (int nst = 4; nst >= 2; --nst) {
      const int W = ws[wi];
      const int tab = tab_fixed + W * tab_warp;
      const int64_t ring = static_cast<int64_t>(W) * nst * g.stage_bytes;
      const int64_t total = 1024 + ring + tab + W * nst * 8;
      const int64_t inflight = static_cast<int64_t>(W) * (nst - 1) * g.box_bytes;
      if (total <= kDsplitSmemLimit && inflight > best) {
        best = inflight;
        g.W = W;
        g.nst = nst;
        g.tab_off = static_cast<int>(ring);
        g.bar_off = static_cast<int>(ring + tab);
        g.total = static_cast<int>(total);
      }
    }
  if (best < 0) g.W = 0;
  return g;
}

// The partials' ring, shared by the CTA's consumer warps behind one producer
// warp: as many stages as fit; W consumer warps (at most kPartMaxWarps) such
// that at least 4 boxes are in flight beyond the ones being worked on.
inline PtGeom pt_geom(int n, int ds, int NT) {
  PtGeom g{};
  g.TM = n <= 16 ? 16 / n : 1;
  g.P = g.TM * n;
  g.mtiles = (g.P + 15) / 16;
  g.box_bytes = g.P * ds * 2;
  g.stage_bytes = (g.box_bytes + 1023) / 1024 * 1024;
  const int tab = 2 * NT * 8 * tc_pitch(ds) * 2;
  int nst = (kDsplitSmemLimit - 1024 - tab) / (g.stage_bytes + 16);
  if (nst > 64) nst = 64;
  g.nst = nst;
  g.W = nst - 4 < kPartMaxWarps ? nst - 4 : kPartMaxWarps;
  g.tab_off = nst * g.stage_bytes;
  g.bar_off = g.tab_off + tab;
  g.total = 1024 + g.bar_off + 2 * nst * 8;
  if (g.W < 1) g.W = 0;
  return g;
}

// Per-warp area of the tensor-core finish: bf16 weights [2 tokens][hi, lo][16
// queries][8 NK sources], then the box's partials (at most 16 pairs x 17 floats).
constexpr int kFinPartFloats = 16 * (ATTNRES_MAX_QUERIES + 1);
__host__ __device__ inline int fin_warp_bytes(int NK) { return 2 * 2 * 16 * 8 * NK * 2 + kFinPartFloats * 4; }
inline PtGeom fin_geom(int n, int ds) { return ring_geom(n, ds, 0, fin_warp_bytes((n + 7) / 8)); }

// The shard as a 4-d tensor (feature within a 64-feature chunk, source,
// token, chunk) and the box {64, n, TM, d_s / 64}, 128-byte swizzle.
bool encode_shard_map(const DsplitArgs& a, const PtGeom& g, CUtensorMap* map) {
  PFN_cuTensorMapEncodeTiled_v12000 fn = tensor_map_encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[4] = {64, static_cast<cuuint64_t>(a.n_src), static_cast<cuuint64_t>(a.T),
                              static_cast<cuuint64_t>(a.d_shard / 64)};
  const cuuint64_t strides[3] = {static_cast<cuuint64_t>(a.src_stride) * 2, static_cast<cuuint64_t>(a.d_shard) * 2,
                                 128};
  const cuuint32_t box[4] = {64, static_cast<cuuint32_t>(a.n_src), static_cast<cuuint32_t>(g.TM),
                             static_cast<cuuint32_t>(a.d_shard / 64)};
  const cuuint32_t es[4] = {1, 1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(a.Src), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

__device__ unsigned int g_dsplit_timeout = 0;

__device__ __forceinline__ void tma_load_box(uint32_t dst, const CUtensorMap* map, int tok0, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, "
      "%5}], [%6];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(0), "r"(0), "r"(tok0), "r"(0), "r"(bar)
      : "memory");
}

// Fire-and-forget fp32 add to global memory (one add per address and launch,
// so the result does not depend on the order of the adds).
__device__ __forceinline__ void red_add(float* p, float v) {
  asm volatile("red.global.add.f32 [%0], %1;" ::"l"(p), "f"(v) : "memory");
}

// Orders this thread's earlier shared-memory accesses (generic proxy) before
// its later async-proxy (TMA) writes to the same memory.
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

template <int NT>
__global__ void __launch_bounds__(kPartMaxWarps * 32 + 32, 1)
    dsplit_partials_tc_kernel(DsplitArgs a, PtGeom G, const __grid_constant__ CUtensorMap tmap) {
  extern __shared__ __align__(16) unsigned char dsm_raw[];
  unsigned char* dsm = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(dsm_raw) + 1023) & ~uintptr_t(1023));
  const int S = a.S, ds = a.d_shard, n = a.n_src;
  const int pitch = tc_pitch(ds);
  bf16* whi = reinterpret_cast<bf16*>(dsm + G.tab_off);  // [NT * 8][pitch]
  bf16* wlo = whi + NT * 8 * pitch;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int W = G.W;  // consumer warps; warp W is the producer
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(dsm + G.bar_off);  // [nst]
  uint64_t* empty_bar = full_bar + G.nst;                              // [nst]
  const uint32_t ring = smem_u32(dsm);
  const int64_t ntiles = (a.T + G.TM - 1) / G.TM;
  // This CTA's boxes: tile blockIdx.x + i * gridDim.x for i < nmine; box i
  // sits in slot i % nst and is taken by consumer warp i % W.
  const int64_t nmine = blockIdx.x < ntiles ? (ntiles - blockIdx.x + gridDim.x - 1) / gridDim.x : 0;
  pdl_trigger();
  pdl_wait();
  if (threadIdx.x == 0) {
    for (int j = 0; j < G.nst; ++j) {
      mbar_init(smem_u32(&full_bar[j]), 1);
      mbar_init(smem_u32(&empty_bar[j]), 1);
    }
    mbar_fence_init();
  }
  __syncthreads();
  if (warp == W) {
    // ------------------------------------------------------------ producer
    if (lane != 0) return;
    bool pok = true;
    int64_t issued = 0;
    for (int64_t i = 0; i < nmine; ++i) {
      const int slot = static_cast<int>(i % G.nst);
      // A fresh barrier counts its (virtual) previous phase as complete.
      if (!mbar_wait(smem_u32(&empty_bar[slot]), static_cast<uint32_t>(((i / G.nst) & 1) ^ 1))) {
        pok = false;
        break;
      }
      const int64_t tile = blockIdx.x + i * gridDim.x;
      mbar_arrive_expect_tx(smem_u32(&full_bar[slot]), G.box_bytes);
      tma_load_box(ring + slot * G.stage_bytes, &tmap, static_cast<int>(tile * G.TM), smem_u32(&full_bar[slot]));
      ++issued;
    }
    if (!pok) {
      atomicOr(&g_dsplit_timeout, 1u);
      // Let the copies still in flight land before the CTA's memory goes.
      for (int64_t i = issued > G.nst ? issued - G.nst : 0; i < issued; ++i)
        (void)mbar_wait(smem_u32(&full_bar[i % G.nst]), static_cast<uint32_t>((i / G.nst) & 1));
    }
    return;
  }
  // The tables, 4 features per thread and step (loads of all steps issued
  // first), by the consumer warps while the first boxes stream in.
  const int nct = W * 32;
  for (int e0 = threadIdx.x * 4; e0 < NT * 8 * ds; e0 += nct * 4 * 4) {
    float w[4][4], gm[4][4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int e = e0 + u * nct * 4, j = e / ds;
      if (e < NT * 8 * ds && j < S) {
        ldg4(a.W + e, w[u]);
        ldg4(a.Gamma + e, gm[u]);
      } else {
        w[u][0] = w[u][1] = w[u][2] = w[u][3] = 0.f;
        gm[u][0] = gm[u][1] = gm[u][2] = gm[u][3] = 0.f;
      }
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int e = e0 + u * nct * 4, j = e / ds, k = e - j * ds;
      if (e >= NT * 8 * ds) continue;
      float hi[4], lo[4];
#pragma unroll
      for (int v = 0; v < 4; ++v) {
        const float x = w[u][v] * gm[u][v];
        hi[v] = __bfloat162float(__float2bfloat16_rn(x));
        lo[v] = x - hi[v];
      }
      st4(whi + j * pitch + k, hi);
      st4(wlo + j * pitch + k, lo);
    }
  }
  named_sync(1, nct);

  const int g = lane >> 2, q = lane & 3;
  const int sg = ((g & 1) << 2) | (g >> 1);  // pair of MMA row g within a 16-pair tile
  const int nsteps = ds / 32;
  bool ok = true;
  for (int64_t i = warp; i < nmine; i += W) {
    const int64_t tile = blockIdx.x + i * gridDim.x;
    const int slot = static_cast<int>(i % G.nst);
    if (!mbar_wait(smem_u32(&full_bar[slot]), static_cast<uint32_t>((i / G.nst) & 1))) {
      ok = false;
      break;
    }
    const uint32_t box = ring + slot * G.stage_bytes;
    for (int mt = 0; mt < G.mtiles; ++mt) {
      // Line of this lane's two pairs in chunk 0, and the chunk stride.
      int L[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) L[h] = min(mt * 16 + sg + 8 * h, G.P - 1);
      float ch[NT][4], cl[NT][4], sq[2][4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) ch[nt][e] = cl[nt][e] = 0.f;
        sq[0][e] = sq[1][e] = 0.f;
      }
      for (int s0 = 0; s0 < nsteps; s0 += 4) {
        uint4 x[4][2];
#pragma unroll
        for (int u = 0; u < 4; ++u)
          if (s0 + u < nsteps) {
            const int s = s0 + u, unit = ((s & 1) << 2) | q;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const int Ls = L[h] + (s >> 1) * G.P;
              const uint32_t addr = (box + Ls * 128u + ((Ls & 7) << 4)) ^ (unit << 4);
              asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                           : "=r"(x[u][h].x), "=r"(x[u][h].y), "=r"(x[u][h].z), "=r"(x[u][h].w)
                           : "r"(addr));
            }
          }
#pragma unroll
        for (int u = 0; u < 4; ++u)
          if (s0 + u < nsteps) {
            // Lane (g, q) holds features 8q' .. 8q' + 7 (q' = the 16-byte
            // unit of this step) of its two pairs: features 8q' + {0,1} |
            // {2,3} are the first MMA's k pairs 2q and 2q + 8, 8q' + {4,5} |
            // {6,7} the second's; the tables are read at the same features.
            const uint32_t A1[4] = {x[u][0].x, x[u][1].x, x[u][0].y, x[u][1].y};
            const uint32_t A2[4] = {x[u][0].z, x[u][1].z, x[u][0].w, x[u][1].w};
            const int kk = (s0 + u) * 32 + q * 8;
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
              const uint4 bh = *reinterpret_cast<const uint4*>(whi + (nt * 8 + g) * pitch + kk);
              const uint4 bl = *reinterpret_cast<const uint4*>(wlo + (nt * 8 + g) * pitch + kk);
              mma16816(ch[nt], A1, bh.x, bh.y);
              mma16816(cl[nt], A1, bl.x, bl.y);
              mma16816(ch[nt], A2, bh.z, bh.w);
              mma16816(cl[nt], A2, bl.z, bl.w);
            }
            // A A^T: B = the A fragments of rows 0..7 (then 8..15) as
            // columns; its diagonal is sum v^2 of each row (bf16 products
            // are exact in fp32).
            mma16816(sq[0], A1, A1[0], A1[2]);
            mma16816(sq[1], A1, A1[1], A1[3]);
            mma16816(sq[0], A2, A2[0], A2[2]);
            mma16816(sq[1], A2, A2[1], A2[3]);
          }
      }
      // Diagonal of A A^T: row g sits at column g of the first block (lane
      // q = g / 2, element g & 1), row g + 8 at column g of the second (rows
      // g + 8: elements 2 + (g & 1)); lane (g, g / 2) holds both.
      const int src_lane = (g << 2) | (g >> 1);
      const float d0 = __shfl_sync(0xffffffffu, (g & 1) ? sq[0][1] : sq[0][0], src_lane);
      const float d1 = __shfl_sync(0xffffffffu, (g & 1) ? sq[1][3] : sq[1][2], src_lane);
      const float ssv[2] = {d0, d1};
      // D fragments: MMA rows g, g + 8 (pairs sg, sg + 8); queries nt * 8 + 2q + {0, 1}.
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int p = mt * 16 + sg + 8 * h;
        if (p >= G.P || tile * G.TM + p / n >= a.T) continue;
        float* prt = a.partials + (tile * G.P + p) * (S + 1);
        if (a.accumulate) {
          if (q == 0) red_add(prt, ssv[h]);
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const int jj = nt * 8 + 2 * q + e;
              if (jj < S) red_add(prt + 1 + jj, ch[nt][2 * h + e] + cl[nt][2 * h + e]);
            }
        } else {
          if (q == 0) prt[0] = ssv[h];
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const int jj = nt * 8 + 2 * q + e;
              if (jj < S) prt[1 + jj] = ch[nt][2 * h + e] + cl[nt][2 * h + e];
            }
        }
      }
    }
    // The slot is free once every lane has read it.
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&empty_bar[slot]));
  }
  // A consumer that gave up leaves its slot held; the producer's own wait
  // then runs out too and drains the copies in flight.
  if (!ok && lane == 0) atomicOr(&g_dsplit_timeout, 1u);
}

// bf16 finish on the tensor cores (n <= 16 sources, shard width a multiple of
// 64). Same boxes and per-warp rings as the tensor-core partials. For each
// token the lanes turn its partials into the softmax weights and write them as
// bf16 hi + lo parts; then per 8 features one MMA (per 8 sources) forms all
// queries' sums: A = the weights (rows: 16 queries; k: the 8 sources' hi
// parts, then their lo parts), B = the sources' 8 features (k: the 8 sources,
// twice), read with ldmatrix.trans from the swizzled box (the 8 source lines
// of a token are 8 consecutive lines, so their units fall in 8 banks).
template <int NK, int R, int kTT>
__global__ void __launch_bounds__(8 * 32, 1)
    dsplit_finish_tc_kernel(DsplitArgs a, PtGeom G, const __grid_constant__ CUtensorMap tmap) {
  extern __shared__ __align__(16) unsigned char dsm_raw[];
  unsigned char* dsm = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(dsm_raw) + 1023) & ~uintptr_t(1023));
  constexpr int np = 8 * NK;
  const int S = a.S, ds = a.d_shard, n = a.n_src;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, q = lane & 3;
  unsigned char* area = dsm + G.tab_off + warp * fin_warp_bytes(NK);
  bf16* wts = reinterpret_cast<bf16*>(area);  // per token of a pair: hi [16][np], then lo [16][np]
  float* part = reinterpret_cast<float*>(area + 2 * 2 * 16 * np * 2);
  uint64_t* bars = reinterpret_cast<uint64_t*>(dsm + G.bar_off) + warp * G.nst;
  const uint32_t ring = smem_u32(dsm + static_cast<size_t>(warp) * G.nst * G.stage_bytes);
  const int64_t ntiles = (a.T + G.TM - 1) / G.TM;
  const int64_t tstride = static_cast<int64_t>(gridDim.x) * G.W;
  const int64_t first = static_cast<int64_t>(blockIdx.x) * G.W + warp;
  const int pf = G.P * (S + 1);  // partial floats of a box
  const float inv_d = 1.0f / static_cast<float>(a.d_total);
  pdl_trigger();
  pdl_wait();
  if (lane == 0) {
    for (int j = 0; j < G.nst; ++j) mbar_init(smem_u32(&bars[j]), 1);
    mbar_fence_init();
    for (int j = 0; j < G.nst; ++j) {
      const int64_t tile = first + j * tstride;
      if (tile >= ntiles) break;
      mbar_arrive_expect_tx(smem_u32(&bars[j]), G.box_bytes);
      tma_load_box(ring + j * G.stage_bytes, &tmap, static_cast<int>(tile * G.TM), smem_u32(&bars[j]));
    }
  }
  // Weights of absent queries and sources stay zero.
  for (int e = lane; e < 2 * 2 * 16 * np; e += 32) wts[e] = __float2bfloat16_rn(0.f);
  // The first box's partials (later boxes' are loaded one box ahead).
  constexpr int kPL = (kFinPartFloats + 31) / 32;
  float pv[kPL];
  auto load_part = [&](int64_t tile) {
    const float* src = a.partials + tile * pf;
    const int64_t left = (a.T * n - tile * G.P) * (S + 1);  // floats that exist from the box's first
#pragma unroll
    for (int r = 0; r < kPL; ++r) {
      const int e = r * 32 + lane;
      if (e < pf && e < left) pv[r] = src[e];
    }
  };
  if (first < ntiles) load_part(first);
  __syncwarp();

  int Q2 = 1;
  while (Q2 < S) Q2 <<= 1;
  const int G2 = 32 / Q2, jq = lane & (Q2 - 1), grp = lane / Q2;
  // Output rows of this lane's D fragments: queries g and g + 8.
  bf16* o0 = nullptr;
  bf16* o1 = nullptr;
#pragma unroll
  for (int jj = 0; jj < ATTNRES_MAX_QUERIES; ++jj) {
    if (jj < S && jj == g) o0 = static_cast<bf16*>(a.out[jj]);
    if (jj < S && jj == g + 8) o1 = static_cast<bf16*>(a.out[jj]);
  }
  bool ok = true;
  int64_t j = 0;
  for (;; ++j) {
    const int64_t tile = first + j * tstride;
    if (tile >= ntiles) break;
    // Park this box's partials in shared memory, then fetch the next box's.
#pragma unroll
    for (int r = 0; r < kPL; ++r)
      if (r * 32 + lane < pf) part[r * 32 + lane] = pv[r];
    if (tile + tstride < ntiles) load_part(tile + tstride);
    const int slot = static_cast<int>(j % G.nst);
    if (!mbar_wait(smem_u32(&bars[slot]), static_cast<uint32_t>((j / G.nst) & 1))) {
      ok = false;
      break;
    }
    __syncwarp();
    const uint32_t box = ring + slot * G.stage_bytes;
    // kTT tokens of the box at a time (independent work to interleave; with
    // two, the second repeats the first when the box or T has no second).
    for (int tm0 = 0; tm0 < G.TM; tm0 += kTT) {
      const int64_t t0 = tile * G.TM + tm0;
      if (t0 >= a.T) break;
      const bool has1 = kTT == 2 && tm0 + 1 < G.TM && t0 + 1 < a.T;
      const int tmv[2] = {tm0, has1 ? tm0 + 1 : tm0};
      // Softmax weights of each token: lane (group, j) takes query j over
      // sources group, group + G2, ...; butterflies combine the groups.
      float m[2] = {-INFINITY, -INFINITY}, ev[2][R];
#pragma unroll
      for (int tt = 0; tt < kTT; ++tt) {
        const float* pt = part + tmv[tt] * n * (S + 1);
#pragma unroll
        for (int r = 0; r < R; ++r) {
          const int i = grp + r * G2;
          ev[tt][r] = -INFINITY;
          if (jq < S && i < n) {
            ev[tt][r] = pt[i * (S + 1) + 1 + jq] * rsqrtf(pt[i * (S + 1)] * inv_d + a.eps);
            m[tt] = fmaxf(m[tt], ev[tt][r]);
          }
        }
      }
      for (int o = Q2; o < 32; o <<= 1) {
        m[0] = fmaxf(m[0], __shfl_xor_sync(0xffffffffu, m[0], o));
        if (kTT == 2) m[1] = fmaxf(m[1], __shfl_xor_sync(0xffffffffu, m[1], o));
      }
      float z[2] = {0.f, 0.f};
#pragma unroll
      for (int tt = 0; tt < kTT; ++tt)
#pragma unroll
        for (int r = 0; r < R; ++r) {
          ev[tt][r] = (jq < S && grp + r * G2 < n) ? __expf(ev[tt][r] - m[tt]) : 0.f;
          z[tt] += ev[tt][r];
        }
      for (int o = Q2; o < 32; o <<= 1) {
        z[0] += __shfl_xor_sync(0xffffffffu, z[0], o);
        if (kTT == 2) z[1] += __shfl_xor_sync(0xffffffffu, z[1], o);
      }
#pragma unroll
      for (int tt = 0; tt < kTT; ++tt) {
        const float inv = 1.0f / z[tt];
        bf16* whi = wts + tt * 2 * 16 * np;
        bf16* wlo = whi + 16 * np;
#pragma unroll
        for (int r = 0; r < R; ++r) {
          const int i = grp + r * G2;
          if (jq < S && i < n) {
            const float w = ev[tt][r] * inv;
            const bf16 h = __float2bfloat16_rn(w);
            whi[jq * np + i] = h;
            wlo[jq * np + i] = __float2bfloat16_rn(w - __bfloat162float(h));
          }
        }
        if (a.lse && grp == 0 && jq < S && (tt == 0 || has1)) a.lse[jq * a.T + t0 + tt] = m[tt] + __logf(z[tt]);
      }
      __syncwarp();
      uint32_t af[2][NK][4];
      int Lsrc[2][NK];
#pragma unroll
      for (int tt = 0; tt < kTT; ++tt) {
        const bf16* whi = wts + tt * 2 * 16 * np;
        const bf16* wlo = whi + 16 * np;
#pragma unroll
        for (int kb = 0; kb < NK; ++kb) {
          af[tt][kb][0] = *reinterpret_cast<const uint32_t*>(whi + g * np + 8 * kb + 2 * q);
          af[tt][kb][1] = *reinterpret_cast<const uint32_t*>(whi + (g + 8) * np + 8 * kb + 2 * q);
          af[tt][kb][2] = *reinterpret_cast<const uint32_t*>(wlo + g * np + 8 * kb + 2 * q);
          af[tt][kb][3] = *reinterpret_cast<const uint32_t*>(wlo + (g + 8) * np + 8 * kb + 2 * q);
          // ldmatrix rows: lane l gives source 8 kb + (l & 7) (clamped to a
          // real one; its weight is zero) of unit 4 uq + (l >> 3).
          Lsrc[tt][kb] = tmv[tt] * n + min(8 * kb + (lane & 7), n - 1);
        }
      }
      for (int c = 0; c < ds / 64; ++c) {
        float acc[2][8][4];
#pragma unroll
        for (int kb = 0; kb < NK; ++kb) {
          uint32_t rr[2][2][4];
#pragma unroll
          for (int tt = 0; tt < kTT; ++tt) {
            const int L = c * G.P + Lsrc[tt][kb];
            const uint32_t lb = box + L * 128u + ((L & 7) << 4);
#pragma unroll
            for (int uq = 0; uq < 2; ++uq) ldsm_x4_trans(lb ^ (((uq << 2) | (lane >> 3)) << 4), rr[tt][uq]);
          }
#pragma unroll
          for (int tt = 0; tt < kTT; ++tt)
#pragma unroll
            for (int uq = 0; uq < 2; ++uq)
#pragma unroll
              for (int mm = 0; mm < 4; ++mm) {
                if (kb == 0)
                  mma16816_z(acc[tt][uq * 4 + mm], af[tt][kb], rr[tt][uq][mm], rr[tt][uq][mm]);
                else
                  mma16816(acc[tt][uq * 4 + mm], af[tt][kb], rr[tt][uq][mm], rr[tt][uq][mm]);
              }
        }
        // D: query g (and g + 8), features c * 64 + 8u + 2q, + 1.
#pragma unroll
        for (int tt = 0; tt < kTT; ++tt) {
          if (tt == 1 && !has1) break;
          const int64_t t = t0 + tt;
          uint32_t* r0 = reinterpret_cast<uint32_t*>(o0 + t * ds + c * 64 + 2 * q);
          uint32_t* r1 = reinterpret_cast<uint32_t*>(o1 + t * ds + c * 64 + 2 * q);
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            if (o0) r0[4 * u] = pack_bf16x2(acc[tt][u][0], acc[tt][u][1]);
            if (o1) r1[4 * u] = pack_bf16x2(acc[tt][u][2], acc[tt][u][3]);
          }
        }
      }
      __syncwarp();
    }
    // The slot is free once every lane has read it: refill it.
    __syncwarp();
    const int64_t next = tile + G.nst * tstride;
    if (lane == 0 && next < ntiles) {
      fence_proxy_async();
      mbar_arrive_expect_tx(smem_u32(&bars[slot]), G.box_bytes);
      tma_load_box(box, &tmap, static_cast<int>(next * G.TM), smem_u32(&bars[slot]));
    }
  }
  if (!ok) {
    if (lane == 0) atomicOr(&g_dsplit_timeout, 1u);
    for (int64_t jj = j; jj < j + G.nst && first + jj * tstride < ntiles; ++jj)
      (void)mbar_wait(smem_u32(&bars[jj % G.nst]), static_cast<uint32_t>((jj / G.nst) & 1));
  }
}

// Raw storage of 4 consecutive features (kept packed in registers until used).
template <typename T> struct Raw4;
template <> struct Raw4<bf16> {
  using type = uint2;
  static constexpr int kBatch = 8;  // sources per load batch (16 registers)
  __device__ static type load(const bf16* p) { return *reinterpret_cast<const uint2*>(p); }
  __device__ static void unpack(type v, float (&x)[4]) {
    x[0] = bf16_lo(v.x); x[1] = bf16_hi(v.x); x[2] = bf16_lo(v.y); x[3] = bf16_hi(v.y);
  }
};
template <> struct Raw4<float> {
  using type = float4;
  static constexpr int kBatch = 4;
  __device__ static type load(const float* p) { return *reinterpret_cast<const float4*>(p); }
  __device__ static void unpack(type v, float (&x)[4]) { x[0] = v.x; x[1] = v.y; x[2] = v.z; x[3] = v.w; }
};

// CH = 4-feature chunks per lane (the shard has at most 128 * CH features);
// QB = the query bound (8 or 16) that sizes the accumulators.
// The work of a warp is a sequence of (token, chunk, batch of sources) items;
// the loads of the next item are issued before the math of the current one,
// so a batch is always in flight, including across the score and softmax
// phase at the start of each token.
template <typename T, int CH, int QB>
__global__ void __launch_bounds__(kDWarps * 32) dsplit_finish_kernel(DsplitArgs a) {
  extern __shared__ __align__(16) float al[];  // [warps][n][Sp] weights
  using R = Raw4<T>;
  constexpr int kB = R::kBatch;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int S = a.S, ds = a.d_shard, n = a.n_src;
  const int Sp = (S + 3) & ~3;
  const int nb = (n + kB - 1) / kB;  // batches per chunk
  const float inv_d = 1.0f / static_cast<float>(a.d_total);
  const int64_t tstride = static_cast<int64_t>(gridDim.x) * kDWarps;
  float* my = al + warp * n * Sp;
  const T* src = static_cast<const T*>(a.Src);
  pdl_trigger();
  pdl_wait();
  int64_t t = static_cast<int64_t>(blockIdx.x) * kDWarps + warp;
  if (t >= a.T) return;
  int c = 0, b = 0;
  auto load_item = [&](int64_t tt, int cc, int bb, typename R::type (&x)[kB]) {
    const int k = (cc * 32 + lane) * 4;
#pragma unroll
    for (int u = 0; u < kB; ++u)
      if (bb * kB + u < n && k < ds) x[u] = R::load(src + (bb * kB + u) * a.src_stride + tt * ds + k);
  };
  float2 acc[QB / 2][4];
  // Lanes of the score phase: Q2 = the power of two >= S, G = 32 / Q2 groups.
  int Q2 = 1;
  while (Q2 < S) Q2 <<= 1;
  const int G = 32 / Q2, jq = lane & (Q2 - 1), grp = lane / Q2;
  auto step = [&](typename R::type (&xc)[kB], typename R::type (&xn)[kB]) -> bool {
    int64_t tn = t;
    int cn = c, bn = b + 1;
    if (bn == nb) {
      bn = 0;
      if (++cn == CH) {
        cn = 0;
        tn += tstride;
      }
    }
    if (tn < a.T) load_item(tn, cn, bn, xn);
    if (c == 0 && b == 0) {
      // Scores and softmax of the token (its partials are contiguous): lane
      // (group, j) takes query j over sources group, group + G, ...; the
      // groups' maxima and sums are then combined by butterflies.
      __syncwarp();
      const float* pt = a.partials + t * n * (S + 1);
      float m = -INFINITY;
      if (jq < S)
        for (int i = grp; i < n; i += G) {
          const float e = pt[i * (S + 1) + 1 + jq] * rsqrtf(pt[i * (S + 1)] * inv_d + a.eps);
          my[i * Sp + jq] = e;
          m = fmaxf(m, e);
        }
      for (int o = Q2; o < 32; o <<= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
      float z = 0.f;
      if (jq < S)
        for (int i = grp; i < n; i += G) {
          const float ez = __expf(my[i * Sp + jq] - m);
          my[i * Sp + jq] = ez;
          z += ez;
        }
      for (int o = Q2; o < 32; o <<= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
      const float inv = 1.0f / z;
      if (jq < S)
        for (int i = grp; i < n; i += G) my[i * Sp + jq] *= inv;
      if (a.lse && grp == 0 && jq < S) a.lse[jq * a.T + t] = m + __logf(z);
      __syncwarp();
    }
    if (b == 0) {
#pragma unroll
      for (int jp = 0; jp < QB / 2; ++jp)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[jp][e] = make_float2(0.f, 0.f);
    }
    // acc[jp][e] = {sum for query 2jp, sum for query 2jp + 1} at feature e:
    // the weight pairs come straight from the 16-byte weight loads and each
    // feature value is duplicated once for all query pairs.
#pragma unroll
    for (int u = 0; u < kB; ++u)
      if (b * kB + u < n) {
        float x[4];
        R::unpack(xc[u], x);
        const float2 xd[4] = {make_float2(x[0], x[0]), make_float2(x[1], x[1]), make_float2(x[2], x[2]),
                              make_float2(x[3], x[3])};
        const float* wr = my + (b * kB + u) * Sp;
#pragma unroll
        for (int j4 = 0; j4 < QB; j4 += 4)
          if (j4 < S) {
            const float4 w4 = *reinterpret_cast<const float4*>(wr + j4);
            const float2 wa = make_float2(w4.x, w4.y), wb = make_float2(w4.z, w4.w);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              acc[j4 / 2][e] = ffma2(wa, xd[e], acc[j4 / 2][e]);
              acc[j4 / 2 + 1][e] = ffma2(wb, xd[e], acc[j4 / 2 + 1][e]);
            }
          }
      }
    if (b == nb - 1) {
      const int k = (c * 32 + lane) * 4;
      if (k < ds) {
#pragma unroll
        for (int j = 0; j < QB; ++j)
          if (j < S) {
            const float2* aj = acc[j / 2];
            const float o[4] = {(j & 1) ? aj[0].y : aj[0].x, (j & 1) ? aj[1].y : aj[1].x,
                                (j & 1) ? aj[2].y : aj[2].x, (j & 1) ? aj[3].y : aj[3].x};
            st4(static_cast<T*>(a.out[j]) + t * ds + k, o);
          }
      }
    }
    t = tn;
    c = cn;
    b = bn;
    return tn < a.T;
  };
  typename R::type xa[kB], xb[kB];
  load_item(t, 0, 0, xa);
  while (step(xa, xb) && step(xb, xa)) {
  }
}

bool finish_on_tensor_cores(const DsplitArgs& a) {
  if (!a.bf16 || a.d_shard % 64 != 0 || a.n_src > 16 || a.T >= (int64_t(1) << 31)) return false;
  return tensor_map_encode_fn() != nullptr && fin_geom(a.n_src, a.d_shard).W >= 1;
}

template <int NK, int R>
cudaError_t launch_finish_tc(const DsplitArgs& a, cudaStream_t s) {
  const PtGeom g = fin_geom(a.n_src, a.d_shard);
  // Boxes of one token (more than 8 sources) take them one at a time.
  auto k = g.TM >= 2 ? dsplit_finish_tc_kernel<NK, R, 2> : dsplit_finish_tc_kernel<NK, R, 1>;
  cudaError_t e = allow_dynamic_smem(reinterpret_cast<const void*>(k), g.total);
  if (e != cudaSuccess) return e;
  alignas(64) CUtensorMap map;
  if (!encode_shard_map(a, g, &map)) return cudaErrorInvalidValue;
  const int64_t tiles = (a.T + g.TM - 1) / g.TM;
  int64_t grid = static_cast<int64_t>(sm_count()) * blocks_per_sm(reinterpret_cast<const void*>(k), g.W * 32, g.total);
  const int64_t need = (tiles + g.W - 1) / g.W;
  if (grid > need) grid = need;
  return launch_pdl(k, static_cast<unsigned>(grid > 0 ? grid : 1), g.W * 32, g.total, s, a, g, map);
}

template <typename T, int CH, int QB>
cudaError_t launch_finish_ch(const DsplitArgs& a, cudaStream_t s) {
  const int smem = finish_smem(a);
  auto k = dsplit_finish_kernel<T, CH, QB>;
  cudaError_t e = allow_dynamic_smem(reinterpret_cast<const void*>(k), smem);
  if (e != cudaSuccess) return e;
  int64_t blocks = (a.T + kDWarps - 1) / kDWarps;
  const int64_t cap = static_cast<int64_t>(sm_count()) * blocks_per_sm(reinterpret_cast<const void*>(k), kDWarps * 32, smem);
  if (blocks > cap) blocks = cap;
  return launch_pdl(k, static_cast<unsigned>(blocks > 0 ? blocks : 1), kDWarps * 32, smem, s, a);
}

template <typename T, int QB>
cudaError_t launch_finish_q(const DsplitArgs& a, cudaStream_t s) {
  const int ch = (a.d_shard + 127) / 128;
  if (ch <= 1) return launch_finish_ch<T, 1, QB>(a, s);
  if (ch <= 2) return launch_finish_ch<T, 2, QB>(a, s);
  if (ch <= 4) return launch_finish_ch<T, 4, QB>(a, s);
  return cudaErrorInvalidValue;
}

template <typename T>
cudaError_t launch_finish_t(const DsplitArgs& a, cudaStream_t s) {
  return a.S <= 8 ? launch_finish_q<T, 8>(a, s) : launch_finish_q<T, 16>(a, s);
}

bool partials_on_tensor_cores(const DsplitArgs& a) {
  if (!a.bf16 || a.d_shard % 64 != 0 || a.n_src > 256 || a.T >= (int64_t(1) << 31)) return false;
  if (!aligned16(a.W) || !aligned16(a.Gamma) || tensor_map_encode_fn() == nullptr) return false;
  return pt_geom(a.n_src, a.d_shard, a.S <= 8 ? 1 : 2).W >= 1;
}

template <int NT>
cudaError_t launch_partials_tc(const DsplitArgs& a, cudaStream_t s) {
  const PtGeom g = pt_geom(a.n_src, a.d_shard, NT);
  auto k = dsplit_partials_tc_kernel<NT>;
  cudaError_t e = allow_dynamic_smem(reinterpret_cast<const void*>(k), g.total);
  if (e != cudaSuccess) return e;
  alignas(64) CUtensorMap map;
  if (!encode_shard_map(a, g, &map)) return cudaErrorInvalidValue;
  const int64_t tiles = (a.T + g.TM - 1) / g.TM;
  const int threads = (g.W + 1) * 32;
  int64_t grid = static_cast<int64_t>(sm_count()) * blocks_per_sm(reinterpret_cast<const void*>(k), threads, g.total);
  const int64_t need = (tiles + g.W - 1) / g.W;
  if (grid > need) grid = need;
  return launch_pdl(k, static_cast<unsigned>(grid > 0 ? grid : 1), threads, g.total, s, a, g, map);
}

}  // namespace

bool dsplit_ok(const DsplitArgs& a) {
  const int es = a.bf16 ? 2 : 4;
  if (a.d_shard % 4 != 0 || a.d_shard > kMaxDsplitShard || a.S < 1 || a.S > ATTNRES_MAX_QUERIES) return false;
  if ((a.d_shard * es) % 8 != 0 || (a.src_stride * es) % 16 != 0 || !aligned16(a.Src)) return false;
  if (finish_smem(a) > 200 * 1024) return false;
  if (static_cast<int64_t>(a.S) * a.d_shard * 4 > 200 * 1024) return false;
  for (int j = 0; j < a.S; ++j)
    if (!aligned16(a.out[j])) return false;
  return true;
}

cudaError_t launch_dsplit_partials(const DsplitArgs& a, cudaStream_t s) {
  if (partials_on_tensor_cores(a)) return a.S <= 8 ? launch_partials_tc<1>(a, s) : launch_partials_tc<2>(a, s);
  const int smem = a.S * a.d_shard * 4;
  const void* fn = a.bf16 ? reinterpret_cast<const void*>(&dsplit_partials_kernel<bf16>)
                          : reinterpret_cast<const void*>(&dsplit_partials_kernel<float>);
  cudaError_t e = allow_dynamic_smem(fn, smem);
  if (e != cudaSuccess) return e;
  int64_t blocks = (static_cast<int64_t>(a.n_src) * a.T + kDWarps - 1) / kDWarps;
  const int64_t cap = static_cast<int64_t>(sm_count()) * blocks_per_sm(fn, kDWarps * 32, smem);
  if (blocks > cap) blocks = cap;
  if (a.bf16) return launch_pdl(dsplit_partials_kernel<bf16>, static_cast<unsigned>(blocks), kDWarps * 32, smem, s, a);
  return launch_pdl(dsplit_partials_kernel<float>, static_cast<unsigned>(blocks), kDWarps * 32, smem, s, a);
}

cudaError_t take_timeout_dsplit(unsigned int* flag) {
  unsigned int zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(flag, g_dsplit_timeout, sizeof(unsigned int));
  if (e != cudaSuccess) return e;
  return cudaMemcpyToSymbol(g_dsplit_timeout, &zero, sizeof(unsigned int));
}

cudaError_t launch_dsplit_finish(const DsplitArgs& a, cudaStream_t s) {
  if (finish_on_tensor_cores(a)) {
    // Sources per lane in the softmax: lanes form 32 / Q2 groups per query
    // (Q2 = the power of two >= S).
    int q2 = 1;
    while (q2 < a.S) q2 <<= 1;
    const int r = (a.n_src + 32 / q2 - 1) / (32 / q2);
    if (a.n_src <= 8) {
      if (r <= 1) return launch_finish_tc<1, 1>(a, s);
      if (r <= 2) return launch_finish_tc<1, 2>(a, s);
      return launch_finish_tc<1, 4>(a, s);
    }
    if (r <= 2) return launch_finish_tc<2, 2>(a, s);
    if (r <= 4) return launch_finish_tc<2, 4>(a, s);
    return launch_finish_tc<2, 8>(a, s);
  }
  return a.bf16 ? launch_finish_t<bf16>(a, s) : launch_finish_t<float>(a, s);
}

}  // namespace attnres
