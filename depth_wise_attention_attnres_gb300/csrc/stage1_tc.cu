// Block AttnRes stage 1 on the tensor cores (bf16 storage), warp-specialized.
//
// Same job as stage1.cu (datacamp explainer, "two-stage computation": the S
// pseudo-queries of a block against the cross-block sources, each source row
// read once): O_j[t] = sum_i softmax_i(e_ij) v_i[t], lse_j[t] = log sum_i
// exp(e_ij), e_ij = w_j^T RMSNorm_j(v_i[t]) (DepthBench reading notes section
// 2.3 / 2.5).
//
// A tile is the n source rows of TM consecutive tokens (P = TM * n <= 16
// (source, token) pairs); TM is the largest that leaves four tile buffers in
// shared memory (up to eight are kept). Three roles work on different tiles at
// once and hand over through shared memory guarded by mbarriers, with no
// CTA-wide barrier in the steady state:
//   producer warp: one TMA tensor copy per tile (box {64 features, n sources,
//     TM rows, d / 64 chunks} of the [n, T, d] sources). The tile lands as
//     128-byte lines ordered (chunk, row, source) with the 128-byte swizzle,
//     so the 8 pairs an ldmatrix reads at one feature offset sit in 8
//     different bank groups;
//   4 score warps: the scores are a small dense contraction with the pairs as
//     the rows of A (16 x d) and w * gamma as B (d x 8 queries, split into
//     bf16 hi + lo so the product keeps about 16 mantissa bits), run as
//     m16n8k16 MMAs with fp32 accumulation; the sums of squares come from the
//     same A fragments as the diagonal of A A^T. A round fills the 16 MMA rows:
//     one tile when P > 8, two consecutive tiles when P <= 8 (w * gamma is then
//     loaded once per k-step for both). The warps split d by 64-feature
//     chunks; their partials meet in shared memory, then a group of lanes per
//     (row, query) takes the softmax over depth with shuffles and writes the
//     weights (double-buffered) and lse;
//   8 output warps, tile by tile: the S weighted sums of every row. With many
//     sources and queries (S * n > 24) they run on the tensor cores: per row,
//     D[16 features x 8 queries] = V^T W, A = V^T taken from the tile with
//     ldmatrix.trans and K holding the 8 sources twice against the weights'
//     bf16 hi and lo parts, D transposed two chunks at a time into a small
//     staging area (one row per query) with stmatrix.trans and written with
//     16-byte stores. With few of them the CUDA cores are cheaper: 8 features
//     per thread, packed fp32x2 FMAs.
// Only the S queries' rows of w * gamma and of the staging are kept, so that
// wide rows (d = 2048) still leave room for four or more tile buffers.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <math.h>

#include "common.cuh"
#include "internal.h"

namespace attnres {
namespace {

__device__ unsigned int g_stage1tc_timeout = 0;

constexpr int kSW = 4;                              // score warps
constexpr int kOW = 8;                              // output warps
constexpr int kScoreThreads = kSW * kWarp;
constexpr int kOutThreads = kOW * kWarp;
constexpr int kThreads = (kSW + kOW + 1) * kWarp;   // + producer warp
constexpr int kMaxPairs = 16;                       // pairs of a tile: one m16 MMA tile
constexpr int kQ = 8;                               // MMA query columns (queries >= S are zero)
constexpr int kF = 8;                               // features per thread on the CUDA-core output path
constexpr int kMaxBuf = 8;                          // tile buffers
constexpr int kBarBytes = 256;
constexpr int kSmemLimit = 227 * 1024;
constexpr int kBtBytes = 16 * 256;                  // MMA weight fragments of a tile: TM * ceil(n / 8) <= 16 blocks
// Weight buffers between the score and output warps: tile it uses buffer
// it % slots. Two suffice for one-tile score rounds; two-tile rounds (P <= 8)
// get four, so the score warps can fill the next round's while the output
// warps still read the last round's.
constexpr int kWSlots = 4;  // the most
inline int weight_slots(int P) { return P <= 8 ? 4 : 2; }
constexpr int kStgPitch = 2 * 128 + 16;             // output staging row: two 64-feature chunks, padded
// full + empty per buffer, the weight handovers each way, then the abort flag
static_assert((2 * kMaxBuf + 2 * kWSlots) * 8 + 4 <= kBarBytes, "barrier area too small");

struct TcGeom {
  int npair;       // pairs a tile holds (TM * n <= 16)
  int TM;          // tokens per tile
  int P;           // pairs of a tile (TM * n)
  int pitch;       // bytes between the rows of w * gamma (d * 2 + 16)
  int srows;       // staging rows per output warp: the S queries (+ one row that absorbs unused ones)
  int buf_bytes;   // one tile buffer (npair rows of d bf16 in swizzled 128-byte lines)
  int nbuf;        // tile buffers
  int w_off, red_off, al_off, bt_off, stg_off, buf_off, total;
};

inline int round_up(int x, int m) { return (x + m - 1) / m * m; }

// The fixed areas hold only what the S queries need: the hi and lo rows of
// w * gamma of each query (2S rows) and S staging rows per output warp.
inline TcGeom tc_geom_for(int n, int d, int S, int TM) {
  TcGeom g{};
  g.TM = TM;
  g.P = TM * n;
  g.npair = g.P;
  g.pitch = d * 2 + 16;
  g.srows = S < kQ ? S + 1 : kQ;
  g.w_off = kBarBytes;                                  // bf16 hi rows [S], then lo rows [S]
  g.red_off = g.w_off + 2 * S * g.pitch;                // fp32 [16][S + 1][kSW] partials
  const int ws = weight_slots(g.P);
  g.al_off = g.red_off + kSW * kMaxPairs * (S + 1) * 4;  // float2 [ws][npair][S2] weights as (a, a)
  g.bt_off = g.al_off + ws * g.npair * round_up(S, 2) * 8;  // bf16 MMA weight fragments [ws][kBtBytes]
  g.stg_off = g.bt_off + ws * kBtBytes;                 // bf16 [kOW][srows][kStgPitch] output staging
  g.buf_off = round_up(g.stg_off + kOW * g.srows * kStgPitch, 1024);
  g.buf_bytes = g.npair * d * 2;
  g.nbuf = (kSmemLimit - 1024 - g.buf_off) / g.buf_bytes;  // 1 KB slack to align the base
  if (g.nbuf > kMaxBuf) g.nbuf = kMaxBuf;
  g.total = g.buf_off + g.nbuf * g.buf_bytes + 1024;
  return g;
}

// The most tokens per tile (at most 16 pairs) that leave four buffers, so
// that the score and output roles each hold one while two more load; else
// one token per tile with as many buffers as fit.
inline TcGeom tc_geom(int n, int d, int S) {
  for (int TM = kMaxPairs / n; TM > 1; --TM) {
    const TcGeom g = tc_geom_for(n, d, S, TM);
    if (g.nbuf >= 4) return g;
  }
  return tc_geom_for(n, d, S, 1);
}

// Which output path a launch takes (the tensor cores pay off from about 24
// multiply-adds per feature and row: measured at d = 2048, S = 6, n = 5).
inline bool outputs_on_tensor_cores(int n, int S) { return S * n > 24; }

// The whole tile in one tensor copy; completion is signalled on `bar`.
__device__ __forceinline__ void tma_load_tile(uint32_t dst, const CUtensorMap* map, int row0, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, "
      "%5}], [%6];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(0), "r"(0), "r"(row0), "r"(0), "r"(bar)
      : "memory");
}

// Shared address of 128-byte line L of a 1 KB-aligned tile with its swizzle
// phase folded in: the 16-byte unit u of the line is then at line_base ^ (u << 4)
// (the swizzle stores unit u at u ^ (L & 7) and only touches address bits 4..6).
__device__ __forceinline__ uint32_t line_base(uint32_t tile, int L) {
  return tile + static_cast<uint32_t>(L) * 128u + static_cast<uint32_t>((L & 7) << 4);
}

// kKT: tiles per score round (2 when a tile has at most 8 pairs, else 1), a
// template parameter so the one-tile instances carry none of the two-tile
// bookkeeping.
template <int S, bool kTC, int kKT>
__global__ void __launch_bounds__(kThreads, 1)
    stage1_tc_kernel(MultiArgs a, TcGeom g, const __grid_constant__ CUtensorMap tmap) {
  constexpr int S2 = (S + 1) / 2 * 2;  // CUDA-core path: weights as (a, a) pairs, S2 per (token, source)
  constexpr int WS = kKT == 2 ? 4 : 2;  // weight buffers (weight_slots of the launch's P)
  constexpr int SC = S + 1;            // partial columns per pair: sum of squares, then the S dots
  extern __shared__ __align__(128) unsigned char smem[];
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem);  // [kMaxBuf] tile landed
  uint64_t* empty_bar = full_bar + kMaxBuf;                 // [kMaxBuf] tile consumed
  uint64_t* afull = empty_bar + kMaxBuf;                    // [WS] weights ready
  uint64_t* aempty = afull + kWSlots;                       // [WS] weights consumed
  volatile int* abort_flag = reinterpret_cast<volatile int*>(aempty + kWSlots);
  unsigned char* wsm = smem + g.w_off;
  float* red = reinterpret_cast<float*>(smem + g.red_off);  // [16][SC][kSW] partials
  float2* alpha = reinterpret_cast<float2*>(smem + g.al_off);
  unsigned char* btab = smem + g.bt_off;  // [kWSlots][TM][ceil(n/8)][8 queries][4] uint2 {hi pair, lo pair}
  unsigned char* bufs = smem + g.buf_off;
  bufs += (1024u - (smem_u32(bufs) & 1023u)) & 1023u;  // the swizzle wants 1 KB alignment

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int n = a.n_src, d = a.d, TM = g.TM;
  const int P = g.P;  // pair m = r * n + i (token r of the tile, source i)
  const int64_t ntok = a.T;
  const int64_t ntiles_total = (ntok + TM - 1) / TM;
  const int64_t t0 = static_cast<int64_t>(blockIdx.x) * ntiles_total / gridDim.x;
  const int64_t t1 = static_cast<int64_t>(blockIdx.x + 1) * ntiles_total / gridDim.x;
  const int nbuf = g.nbuf;
  const int nchunk = d >> 6;  // 64-feature chunks: one 128-byte line per pair

  pdl_trigger();
  if (tid == 0) {
    for (int b = 0; b < nbuf; ++b) {
      mbar_init(smem_u32(&full_bar[b]), 1);
      mbar_init(smem_u32(&empty_bar[b]), kSW + kOW);
    }
    for (int k = 0; k < WS; ++k) {
      mbar_init(smem_u32(&afull[k]), kSW);
      mbar_init(smem_u32(&aempty[k]), kOW);
    }
    *reinterpret_cast<int*>(aempty + kWSlots) = 0;
    mbar_fence_init();
  }
  __syncthreads();
  pdl_wait();  // everything below may read what the previous kernel wrote

  bool ok = true;
  if (warp == kSW + kOW) {
    // ------------------------------------------------------------ producer
    if (lane != 0) return;
    const uint32_t box_bytes = static_cast<uint32_t>(P) * static_cast<uint32_t>(d) * 2u;
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap)) : "memory");
    int b = 0;
    uint32_t phase = 0;
    int64_t issued = 0;
    for (int64_t tile = t0; tile < t1; ++tile) {
      // A fresh barrier counts its (virtual) previous phase as complete, so
      // the first round of waits on parity 1 passes at once.
      if (!mbar_wait(smem_u32(&empty_bar[b]), phase ^ 1u)) {
        ok = false;
        break;
      }
      // Rows past T are zero-filled; the transaction always counts the whole box.
      const uint32_t fb = smem_u32(&full_bar[b]);
      if (issued != a.withhold) {  // the test hook leaves this buffer unfilled
        mbar_arrive_expect_tx(fb, box_bytes);
        tma_load_tile(smem_u32(bufs + b * g.buf_bytes), &tmap, static_cast<int>(tile * TM), fb);
      }
      ++issued;
      if (++b == nbuf) {
        b = 0;
        phase ^= 1u;
      }
    }
    if (!ok) {
      atomicOr(&g_stage1tc_timeout, 1u);
      // Let the copies still in flight land before this CTA's memory goes
      // (a withheld copy was never issued).
      for (int64_t it = issued > nbuf ? issued - nbuf : 0; it < issued; ++it)
        if (it != a.withhold)
          (void)mbar_wait(smem_u32(&full_bar[it % nbuf]), static_cast<uint32_t>((it / nbuf) & 1));
    }
    return;
  }

  // w * gamma as bf16 hi + lo rows (row q: hi part of query q, row S + q:
  // its lo part), by the score and output warps while the producer already
  // fills the pipeline; loads are issued in groups of four per thread before
  // any of them is used.
  {
    constexpr int kCT = kScoreThreads + kOutThreads;
    const int nv = S * d / 4;
    for (int base = tid; base < nv; base += 4 * kCT) {
      float4 wv[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int v = base + u * kCT;
        wv[u] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (v < nv) {
          const float4 x = *reinterpret_cast<const float4*>(a.W + v * 4);
          const float4 y = *reinterpret_cast<const float4*>(a.Gamma + v * 4);
          wv[u] = make_float4(x.x * y.x, x.y * y.y, x.z * y.z, x.w * y.w);
        }
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int v = base + u * kCT;
        if (v < nv) {
          const int q = (v * 4) / d, k = v * 4 - q * d;
          const float w[4] = {wv[u].x, wv[u].y, wv[u].z, wv[u].w};
          float hi[4], lo[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            hi[e] = __bfloat162float(__float2bfloat16_rn(w[e]));
            lo[e] = w[e] - hi[e];
          }
          st4(reinterpret_cast<bf16*>(wsm + q * g.pitch) + k, hi);
          st4(reinterpret_cast<bf16*>(wsm + (S + q) * g.pitch) + k, lo);
        }
      }
    }
    // MMA weight fragments of sources >= n and of queries >= S stay zero.
    for (int v = tid; v < WS * kBtBytes / 16; v += kCT) reinterpret_cast<uint4*>(btab)[v] = make_uint4(0u, 0u, 0u, 0u);
    named_sync(2, kCT);
  }

  if (warp < kSW) {
    // ------------------------------------------------------------- scores
    // The scores of a round are one m16 MMA tile: with P > 8 pairs a tile
    // fills it alone; with P <= 8 two consecutive tiles share it (rows 0-7
    // the first tile's pairs, rows 8-15 the second's), so w * gamma is loaded
    // once per k-step for both and the MMA chains are twice as productive.
    const float inv_d = 1.0f / static_cast<float>(d);
    const int cb = warp * nchunk / kSW, ce = (warp + 1) * nchunk / kSW;  // this warp's chunks
    constexpr int KT = kKT;          // tiles per round
    const int RP = KT == 2 ? 8 : P;  // MMA rows per tile
    const int a_row = (lane & 7) + ((lane >> 3) & 1) * 8;
    const int a_koff = (lane >> 4) * 8;
    const int a_tile = a_row / RP;                             // which tile of the round this row reads
    const int a_pair = a_row - a_tile * RP;
    // Hi rows, then lo rows. Lanes of queries >= S read query 0's rows: what
    // they feed lands only in the MMA columns of queries >= S, never read.
    const int b_row = ((lane & 7) < S ? (lane & 7) : 0) + ((lane >> 4) & 1) * S;
    const int b_koff = ((lane >> 3) & 1) * 8;
    const uint32_t b_base = smem_u32(wsm + b_row * g.pitch) + (cb * 64 + b_koff) * 2;
    const uint32_t a_x = static_cast<uint32_t>(a_koff) * 2u;  // this lane's 16-byte unit within a k-step
    const int gid = lane >> 2, tig = lane & 3;
    // Softmax: a group of G lanes (n rounded up to a power of two) per (token, query).
    int lgG = 0;
    while ((1 << lgG) < n) ++lgG;
    const int G = 1 << lgG;
    const int nk = (n + 7) >> 3;
    const int TMS = TM * S;
    const int64_t ntile = t1 - t0;
    int b = 0;            // buffer of tile it, and the parity of its current use
    uint32_t phase = 0;
    for (int64_t it = 0; it < ntile; it += KT) {
      // Tiles this round (the last round of a CTA may hold one).
      const int kt = KT == 1 ? 1 : static_cast<int>(min(static_cast<int64_t>(KT), ntile - it));
      // Buffers of the round's tiles: b, and the one after it.
      const int bk0 = b;
      const uint32_t ph0 = phase;
      int bk1 = b + 1;
      uint32_t ph1 = phase;
      if (bk1 == nbuf) {
        bk1 = 0;
        ph1 ^= 1u;
      }
      bool got = mbar_wait(smem_u32(&full_bar[bk0]), ph0);
      if (kt == 2) got = got && mbar_wait(smem_u32(&full_bar[bk1]), ph1);
      // A one-tile round also waits here for its weight buffer (measured
      // faster than waiting after the MMAs); a two-tile round waits after
      // them, so its MMAs overlap the output warps' last tile.
      if (KT == 1) got = got && mbar_wait(smem_u32(&aempty[it % WS]), static_cast<uint32_t>(((it / WS) & 1) ^ 1));
      b = kt == 2 ? bk1 : bk0;
      phase = kt == 2 ? ph1 : ph0;
      if (++b == nbuf) {
        b = 0;
        phase ^= 1u;
      }
      // The score warps meet at a named barrier, so giving up is decided jointly.
      if (!got) *abort_flag = 1;
      named_sync(1, kScoreThreads);
      if (*abort_flag) {
        ok = false;
        break;
      }
      // The line this lane reads for MMA row a_row; rows past the round's
      // pairs only pad the m16 tile and read the first pair.
      const bool a_live = a_pair < P && a_tile < kt;
      const uint32_t a_buf = smem_u32(bufs + (a_live && a_tile == 1 ? bk1 : bk0) * g.buf_bytes);
      const int a_p = a_live ? a_pair : 0;
      {
        float sh[4] = {0.f, 0.f, 0.f, 0.f}, sl[4] = {0.f, 0.f, 0.f, 0.f};
        float s0[4] = {0.f, 0.f, 0.f, 0.f}, s1[4] = {0.f, 0.f, 0.f, 0.f};
        // Per chunk: the line of this lane's pair, then its four k-steps (one
        // XOR each). All fragments of a chunk are loaded before its MMAs,
        // since the asm statements issue in program order.
        for (int c = cb; c < ce; ++c) {
          const uint32_t off = line_base(a_buf, c * P + a_p) ^ a_x;
          const uint32_t bo = b_base + static_cast<uint32_t>(c - cb) * 128u;
          uint32_t av[4][4], bv[4][4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            ldsm_x4(off ^ (32u * u), av[u]);
            ldsm_x4(bo + 32u * u, bv[u]);
          }
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            mma16816(sh, av[u], bv[u][0], bv[u][1]);  // hi part of w * gamma
            mma16816(sl, av[u], bv[u][2], bv[u][3]);  // lo part
            mma16816(s0, av[u], av[u][0], av[u][2]);  // A A^T, columns 0..7
            mma16816(s1, av[u], av[u][1], av[u][3]);  // A A^T, columns 8..15
          }
        }
        // This warp is done with the round's tiles.
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(smem_u32(&empty_bar[bk0]));
          if (kt == 2) mbar_arrive(smem_u32(&empty_bar[bk1]));
        }
        // Lane (gid, tig) holds the dots of MMA rows gid, gid + 8 with
        // queries 2 tig, 2 tig + 1; row x of the MMA is row x of red[].
        const bool lo_live = gid < P;
        const bool hi_live = KT == 2 ? (gid < P && kt == 2) : gid + 8 < P;
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int q = 2 * tig + e;
          if (q < S) {
            if (lo_live) red[(gid * SC + 1 + q) * kSW + warp] = sh[e] + sl[e];
            if (hi_live) red[((gid + 8) * SC + 1 + q) * kSW + warp] = sh[2 + e] + sl[2 + e];
          }
        }
        // Diagonal of A A^T: row gid in s0[gid & 1], row gid + 8 in s1[2 + (gid & 1)],
        // held by the lane whose 2 tig + e equals gid (selects keep registers).
        if (tig == (gid >> 1)) {
          const bool odd = gid & 1;
          if (lo_live) red[(gid * SC) * kSW + warp] = odd ? s0[1] : s0[0];
          if (hi_live) red[((gid + 8) * SC) * kSW + warp] = odd ? s1[3] : s1[2];
        }
      }
      // The weight buffers of the round's tiles (tile it + k uses buffer
      // (it + k) % WS) must be free before the softmax writes them.
      if (KT == 2) {
        bool free_ok = true;
        for (int k = 0; k < kt; ++k)
          free_ok = free_ok && mbar_wait(smem_u32(&aempty[(it + k) % WS]),
                                         static_cast<uint32_t>((((it + k) / WS) & 1) ^ 1));
        if (!free_ok) *abort_flag = 1;
      }
      named_sync(1, kScoreThreads);
      if (*abort_flag) {
        ok = false;
        break;
      }
      // Softmax over depth, one lane per source: max and mass by shuffles
      // within the group.
      const int sm_items = kt * TMS * G;
      for (int base = 0; base < sm_items; base += kScoreThreads) {
        const int item = base + tid;
        const int i = item & (G - 1);
        const int krj = item >> lgG;          // (tile of the round, token, query)
        const int k = KT == 2 && krj >= TMS ? 1 : 0;  // a round has at most two tiles
        const int rj = krj - k * TMS;
        const int r = rj / S, j = rj - (rj / S) * S;
        const int64_t row0 = (t0 + it + k) * TM;
        const bool valid = item < sm_items && i < n;
        float e = -INFINITY;
        if (valid) {
          const int p = k * RP + r * n + i;   // row of red[]
          // The four warps' partials of pair p sit side by side.
          const float4 sq = *reinterpret_cast<const float4*>(red + (p * SC) * kSW);
          const float4 dt = *reinterpret_cast<const float4*>(red + (p * SC + 1 + j) * kSW);
          const float ss = ((sq.x + sq.y) + sq.z) + sq.w;
          const float dot = ((dt.x + dt.y) + dt.z) + dt.w;
          e = dot * rsqrtf(ss * inv_d + a.eps);
        }
        // Butterflies over the group (G <= 16; the bound is the same in every
        // lane, so the unrolled steps past it are skipped by the whole warp).
        float mx = e;
#pragma unroll
        for (int off = 1; off < 16; off <<= 1)
          if (off < G) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
        const float x = valid ? __expf(e - mx) : 0.f;
        float z = x;
#pragma unroll
        for (int off = 1; off < 16; off <<= 1)
          if (off < G) z += __shfl_xor_sync(0xffffffffu, z, off);
        if (valid) {
          const int ab = static_cast<int>((it + k) % WS);
          const float wgt = __fdividef(x, z);
          if constexpr (kTC) {
            // B fragment of the output MMA for token r, source block i / 8 and
            // query j: {hi(a[2t]), hi(a[2t+1])}, {lo(a[2t]), lo(a[2t+1])}, t = (i % 8) / 2.
            unsigned char* bt = btab + ab * kBtBytes;
            const bf16 hi = __float2bfloat16_rn(wgt);
            const bf16 lo = __float2bfloat16_rn(wgt - __bfloat162float(hi));
            bf16* ep = reinterpret_cast<bf16*>(bt + (((r * nk + (i >> 3)) * 8 + j) * 4 + ((i & 7) >> 1)) * 8);
            ep[i & 1] = hi;
            ep[2 + (i & 1)] = lo;
          } else {
            float2* al = alpha + ab * g.npair * S2;
            al[(r * n + i) * S2 + j] = make_float2(wgt, wgt);
          }
          if (i == 0 && a.lse && row0 + r < ntok) a.lse[j * ntok + row0 + r] = mx + __logf(z);
        }
      }
      // Weights of the round's tiles are ready: each score warp arrives once
      // its lanes have written theirs (the warp barrier orders the lanes'
      // stores before lane 0's release). red[] is rewritten by the next round
      // only after every score thread has passed the named barrier at its top.
      __syncwarp();
      if (lane == 0)
        for (int k = 0; k < kt; ++k) mbar_arrive(smem_u32(&afull[(it + k) % WS]));
    }
  } else {
    // ------------------------------------------------------------- outputs
    const int ow = warp - kSW;
    int b = 0;
    uint32_t phase = 0;
    int it = 0;
    if constexpr (kTC) {
      // Output warp ow owns a run of chunks. Per token and block of 16
      // features: D[16 features x 8 queries] = A B with A = V^T from
      // ldmatrix.trans (the k columns repeat the 8 sources twice) and B = the
      // weights' bf16 hi parts for k < 8 and lo parts for k >= 8 (one MMA per
      // 8 sources). D goes through stmatrix.trans into the warp's staging rows
      // (one per query), then out with 16-byte stores.
      const int cb = ow * nchunk / kOW, ce = (ow + 1) * nchunk / kOW;
      const int ncw = ce - cb;
      const int f_beg = cb * 64;
      const int nk = (n + 7) >> 3;
      unsigned char* stg = smem + g.stg_off + ow * g.srows * kStgPitch;
      const int l8 = lane & 7, lhalf = (lane >> 3) & 1;
      // Staging row of query l8; queries >= S share the last row, whose
      // contents are never copied out.
      const uint32_t st_base = smem_u32(stg) + (l8 < S ? l8 : g.srows - 1) * kStgPitch + lhalf * 16;
      const uint32_t lx = static_cast<uint32_t>(lhalf) << 4;
      // Copy-out of two chunks (S rows of 16 16-byte pieces): lane l takes
      // pieces l, l + 32, ..., i.e. piece l % 16 of rows l / 16, l / 16 + 2, ...
      // Their output rows and staging offsets are fixed per lane, so they are
      // formed once here rather than per piece.
      constexpr int kPieces = (S * 16 + kWarp - 1) / kWarp;
      bf16* obase[kPieces];
      uint32_t soff[kPieces];
#pragma unroll
      for (int k = 0; k < kPieces; ++k) {
        const int q = (lane >> 4) + 2 * k;
        const int ch = lane & 15;
        obase[k] = q < S ? static_cast<bf16*>(a.out[q]) + f_beg + ch * 8 : nullptr;
        soff[k] = static_cast<uint32_t>(q * kStgPitch + ch * 16);
      }
      for (int64_t tile = t0; tile < t1; ++tile, ++it) {
        const int ab = it % WS;
        const uint32_t aph = static_cast<uint32_t>((it / WS) & 1);
        // Weights ready; waiting on the tile's own barrier as well makes the
        // copied rows visible to this warp.
        const bool got = mbar_wait(smem_u32(&afull[ab]), aph) && mbar_wait(smem_u32(&full_bar[b]), phase);
        if (!__all_sync(0xffffffffu, got)) {
          ok = false;
          break;
        }
        const uint32_t bb = smem_u32(bufs + b * g.buf_bytes);
        const uint2* bt = reinterpret_cast<const uint2*>(btab + ab * kBtBytes);
        const int64_t row0 = tile * TM;
        const int rows = static_cast<int>(min(static_cast<int64_t>(TM), ntok - row0));
        for (int r = 0; r < rows; ++r) {
          uint2 bf[2];
#pragma unroll
          for (int kb = 0; kb < 2; ++kb) bf[kb] = kb < nk ? bt[(r * nk + kb) * 32 + lane] : make_uint2(0u, 0u);
          const int64_t row = row0 + r;
          // Two chunks (8 blocks) at a time: all fragment loads, then the
          // independent MMAs, then the transposing stores into the staging
          // rows, which then go out as 16-byte pieces of 256-byte row runs.
          for (int c = 0; c < ncw; c += 2) {
            float acc[8][4];
#pragma unroll
            for (int u = 0; u < 8; ++u) acc[u][0] = acc[u][1] = acc[u][2] = acc[u][3] = 0.f;
            const bool two = c + 1 < ncw;
#pragma unroll
            for (int kb = 0; kb < 2; ++kb) {
              if (kb < nk) {
                // Lanes past the last source point at source 0; its weights are zero.
                const int i = kb * 8 + l8;
                const int pr = r * n + (i < n ? i : 0);
                uint32_t mv[8][2];
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                  if (h == 0 || two) {
                    const uint32_t off = line_base(bb, (cb + c + h) * P + pr) ^ lx;
#pragma unroll
                    for (int u = 0; u < 4; ++u) ldsm_x2_trans(off ^ (32u * u), mv[h * 4 + u][0], mv[h * 4 + u][1]);
                  }
                }
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                  if (u < 4 || two) {
                    const uint32_t av[4] = {mv[u][0], mv[u][1], mv[u][0], mv[u][1]};
                    mma16816(acc[u], av, bf[kb].x, bf[kb].y);
                  }
                }
              }
            }
            __syncwarp();  // the previous copy-out has read the staging rows
#pragma unroll
            for (int u = 0; u < 8; ++u)
              if (u < 4 || two)
                stsm_x2_trans(st_base + static_cast<uint32_t>(u * 32), pack_bf16x2(acc[u][0], acc[u][1]),
                              pack_bf16x2(acc[u][2], acc[u][3]));
            __syncwarp();
            if (two) {
              const int64_t ro = row * d + c * 64;
#pragma unroll
              for (int k = 0; k < kPieces; ++k) {
                if ((lane >> 4) + 2 * k < S) {
                  const uint4 v = *reinterpret_cast<const uint4*>(stg + soff[k]);
                  *reinterpret_cast<uint4*>(obase[k] + ro) = v;
                }
              }
            } else {
              // The warp's last chunk alone: 8 pieces per row.
              for (int idx = lane; idx < S * 8; idx += kWarp) {
                const int q = idx >> 3;
                const int ch = idx - q * 8;
                const uint4 v = *reinterpret_cast<const uint4*>(stg + q * kStgPitch + ch * 16);
                *reinterpret_cast<uint4*>(static_cast<bf16*>(a.out[q]) + row * d + f_beg + c * 64 + ch * 8) = v;
              }
            }
          }
        }
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(smem_u32(&aempty[ab]));
          mbar_arrive(smem_u32(&empty_bar[b]));
        }
        if (++b == nbuf) {
          b = 0;
          phase ^= 1u;
        }
      }
    } else {
      // Groups of d / 8 threads, one token of the tile per group at a time, 8
      // features per thread, packed fp32x2 FMAs with the weights stored as
      // (a, a) pairs.
      const int otid = tid - kScoreThreads;
      const int tpr = d / kF;
      const int ngrp = kOutThreads / tpr;
      const int grp = otid / tpr;
      const int k = (otid - grp * tpr) * kF;
      const uint32_t kx = static_cast<uint32_t>((k >> 3) & 7) << 4;
      const int kc = k >> 6;
      for (int64_t tile = t0; tile < t1; ++tile, ++it) {
        const int ab = it % WS;
        const uint32_t aph = static_cast<uint32_t>((it / WS) & 1);
        const bool got = mbar_wait(smem_u32(&afull[ab]), aph) && mbar_wait(smem_u32(&full_bar[b]), phase);
        if (!__all_sync(0xffffffffu, got)) {
          ok = false;
          break;
        }
        const uint32_t bb = smem_u32(bufs + b * g.buf_bytes);
        const float2* al = alpha + ab * g.npair * S2;
        const int64_t row0 = tile * TM;
        const int rows = static_cast<int>(min(static_cast<int64_t>(TM), ntok - row0));
        // Threads past the last group idle.
        for (int r = grp < ngrp ? grp : TM; r < rows; r += ngrp) {
          float2 acc[S][kF / 2];
#pragma unroll
          for (int j = 0; j < S; ++j)
#pragma unroll
            for (int e = 0; e < kF / 2; ++e) acc[j][e] = make_float2(0.f, 0.f);
          for (int i = 0; i < n; ++i) {
            uint4 xv;
            asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                         : "=r"(xv.x), "=r"(xv.y), "=r"(xv.z), "=r"(xv.w)
                         : "r"(line_base(bb, kc * P + r * n + i) ^ kx));
            const float2 x2[4] = {make_float2(bf16_lo(xv.x), bf16_hi(xv.x)), make_float2(bf16_lo(xv.y), bf16_hi(xv.y)),
                                  make_float2(bf16_lo(xv.z), bf16_hi(xv.z)), make_float2(bf16_lo(xv.w), bf16_hi(xv.w))};
            const float4* ai = reinterpret_cast<const float4*>(al + (r * n + i) * S2);
#pragma unroll
            for (int jj = 0; jj < S2 / 2; ++jj) {
              const float4 a4 = ai[jj];
              const float2 a0 = make_float2(a4.x, a4.y), a1 = make_float2(a4.z, a4.w);
#pragma unroll
              for (int e = 0; e < kF / 2; ++e) {
                acc[2 * jj][e] = ffma2(a0, x2[e], acc[2 * jj][e]);
                if (2 * jj + 1 < S) acc[2 * jj + 1][e] = ffma2(a1, x2[e], acc[2 * jj + 1][e]);
              }
            }
          }
          const int64_t row = row0 + r;
#pragma unroll
          for (int j = 0; j < S; ++j) {
            const uint4 o = make_uint4(pack_bf16x2(acc[j][0].x, acc[j][0].y), pack_bf16x2(acc[j][1].x, acc[j][1].y),
                                       pack_bf16x2(acc[j][2].x, acc[j][2].y), pack_bf16x2(acc[j][3].x, acc[j][3].y));
            *reinterpret_cast<uint4*>(static_cast<bf16*>(a.out[j]) + row * d + k) = o;
          }
        }
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(smem_u32(&aempty[ab]));
          mbar_arrive(smem_u32(&empty_bar[b]));
        }
        if (++b == nbuf) {
          b = 0;
          phase ^= 1u;
        }
      }
    }
  }
  if (!ok) atomicOr(&g_stage1tc_timeout, 1u);
}

// The sources as a 4-d tensor (feature within chunk, source, token, chunk) and
// the tile box {64, n, TM, d / 64}, 128-byte swizzle.
bool encode_tile_map(const MultiArgs& a, const TcGeom& g, CUtensorMap* map) {
  PFN_cuTensorMapEncodeTiled_v12000 fn = tensor_map_encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[4] = {64, static_cast<cuuint64_t>(a.n_src), static_cast<cuuint64_t>(a.T),
                              static_cast<cuuint64_t>(a.d / 64)};
  const cuuint64_t strides[3] = {static_cast<cuuint64_t>(a.src_stride) * 2, static_cast<cuuint64_t>(a.d) * 2, 128};
  const cuuint32_t box[4] = {64, static_cast<cuuint32_t>(a.n_src), static_cast<cuuint32_t>(g.TM),
                             static_cast<cuuint32_t>(a.d / 64)};
  const cuuint32_t es[4] = {1, 1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(a.V), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int S, bool kTC, int kKT>
cudaError_t launch_s(const MultiArgs& a, const TcGeom& g, cudaStream_t s) {
  auto k = stage1_tc_kernel<S, kTC, kKT>;
  cudaError_t e = allow_dynamic_smem(reinterpret_cast<const void*>(k), g.total);
  if (e != cudaSuccess) return e;
  alignas(64) CUtensorMap map;
  if (!encode_tile_map(a, g, &map)) return cudaErrorInvalidValue;
  const int64_t tiles = (a.T + g.TM - 1) / g.TM;
  int64_t grid = static_cast<int64_t>(sm_count()) * blocks_per_sm(reinterpret_cast<const void*>(k), kThreads, g.total);
  if (grid > tiles) grid = tiles;
  return launch_pdl(k, static_cast<unsigned>(grid), kThreads, g.total, s, a, g, map);
}

template <int S, bool kTC>
cudaError_t launch_kt(const MultiArgs& a, const TcGeom& g, cudaStream_t s) {
  return g.P <= 8 ? launch_s<S, kTC, 2>(a, g, s) : launch_s<S, kTC, 1>(a, g, s);
}

template <int S>
cudaError_t launch_q(const MultiArgs& a, const TcGeom& g, cudaStream_t s) {
  return outputs_on_tensor_cores(a.n_src, S) ? launch_kt<S, true>(a, g, s) : launch_kt<S, false>(a, g, s);
}

}  // namespace

bool stage1_tc_ok(const MultiArgs& a) {
  if (!a.bf16 || a.S < 1 || a.S > kQ || a.n_src < 1 || a.n_src > kMaxPairs) return false;
  if (a.d % 64 != 0 || a.d > kF * kOutThreads || a.T >= (int64_t(1) << 31)) return false;
  if (!aligned16(a.V) || ((a.src_stride * 2) % 16) != 0) return false;
  if (!aligned16(a.W) || !aligned16(a.Gamma)) return false;
  for (int j = 0; j < a.S; ++j)
    if (!aligned16(a.out[j])) return false;
  const TcGeom g = tc_geom(a.n_src, a.d, a.S);
  return g.TM >= 1 && g.nbuf >= 2 && g.total <= kSmemLimit && tensor_map_encode_fn() != nullptr;
}

cudaError_t launch_stage1_tc(const MultiArgs& a, cudaStream_t s) {
  const TcGeom g = tc_geom(a.n_src, a.d, a.S);
  switch (a.S) {
    case 1: return launch_q<1>(a, g, s);
    case 2: return launch_q<2>(a, g, s);
    case 3: return launch_q<3>(a, g, s);
    case 4: return launch_q<4>(a, g, s);
    case 5: return launch_q<5>(a, g, s);
    case 6: return launch_q<6>(a, g, s);
    case 7: return launch_q<7>(a, g, s);
    case 8: return launch_q<8>(a, g, s);
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
