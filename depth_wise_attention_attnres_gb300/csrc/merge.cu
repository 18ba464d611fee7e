// Block AttnRes stage 2 (online-softmax merge) and running-sum kernels.
//
// Merge, per token row (datacamp explainer, "two-stage computation"; the
// running sum of the current block is one more softmax source, DepthBench
// reading notes section 2.5):
//   P   <- P + f_prev                       (fp32 running sum, optional)
//   s_P  = w^T (gamma * P / sqrt(mean(P^2) + eps))
//   M    = max(lse, s_P),  a = exp(lse - M),  b = exp(s_P - M)
//   out  = (a * O + b * P) / (a + b)
// where (O, lse) is the stage-1 read of this sublayer over the cross-block
// sources. Accumulate / freeze (LLMRes blog "Block Attention Residuals": a
// block is represented by the sum of its outputs): P <- P + f, or
// summary <- round(P + f).
//
// Both are HBM-bound streaming kernels (a few flops per byte).
//
// The fast merge uses the same pipeline as the Full read: per CTA a producer
// warp moves tiles of TM consecutive token rows of O, f and P (each tile of
// each stream is one contiguous byte range, so one 1-D bulk copy on the TMA
// engine) into a ring of shared-memory stages guarded by mbarriers; bulk
// copies keep far more bytes in flight than per-thread loads can. Eight
// consumer warps split the tile: 8/TM warps per row, each owning a contiguous
// part of the row, lane l holding its 4-feature chunks l, l+32, ... (8-byte
// bf16 and 16-byte fp32 shared loads, free of bank conflicts). The parts of a
// row combine their two sums through shared memory behind a named barrier of
// just that row's warps. P and out leave with coalesced 16/8-byte stores.
#include <math.h>

#include "common.cuh"
#include "internal.h"

namespace attnres {
namespace {

constexpr int kBlock = 256;
constexpr int kWarps = kBlock / 32;

// ------------------------------------------------------------- fast merge --

__device__ unsigned int g_merge_timeout = 0;

constexpr int kMNW = 8;                      // consumer warps
constexpr int kMThreads = (kMNW + 1) * 32;   // + producer warp
constexpr int kMStages = 3;                   // stages at most (two for 2-row tiles of wide rows)
constexpr int kMBar = 128;                   // barrier area
constexpr int kMStageBudget = 34 * 1024;     // bytes of one stage (TM rows)

struct MergeGeom {
  int TM;          // rows per tile (1, 2, 4 or 8)
  int nst;         // stages (2 or 3)
  int wpr;         // consumer warps per row = 8 / TM
  int stage_bytes;
  int wq_off, red_off, stage_off, total;
};

// A stage holds TM rows of O_j, of each of the q parts and (with a stored
// base) of P. pre: room for gamma_pre next to w * gamma (the pre-norm merge).
inline MergeGeom merge_geom(int d, int es, bool pre, int nparts, bool with_base) {
  MergeGeom g{};
  const int row_bytes = d * (es * (1 + nparts) + (with_base ? 4 : 0));
  g.TM = 8;
  while (g.TM > 1 && g.TM * row_bytes > kMStageBudget) g.TM >>= 1;
  g.nst = kMStages;
  // When tiles twice as tall fit in two stages within the bytes three stages
  // would hold, take them: the consumers' fixed work per tile (the cross-warp
  // sums, the softmax, the barriers) then covers twice the rows. Measured at
  // 131072 x 2048: merge 2 (12 KB rows) 347 -> 315 us, merge 4 (20 KB rows)
  // 719 -> 696 us.
  if (g.TM < 8 && 2 * (2 * g.TM) * row_bytes <= kMStages * kMStageBudget) {
    g.TM *= 2;
    g.nst = 2;
  }
  g.wpr = kMNW / g.TM;
  g.stage_bytes = g.TM * row_bytes;
  g.wq_off = kMBar;
  g.red_off = g.wq_off + (pre ? 2 : 1) * d * 4;
  g.stage_off = (g.red_off + kMNW * 4 * 4 + 127) / 128 * 128;  // [kMNW][3] sums + [kMNW] pre-norm sums
  g.total = g.stage_off + g.nst * g.stage_bytes;
  return g;
}

// Q = 4-feature chunks per lane (a warp covers at most 128 * Q features).
// kPre: also write the sublayer pre-norm of the merged row (a separate
// instance, so the plain merge keeps its own code).
// kSum: also write the block summary (a.summary; a separate instance, so the
// plain merge keeps its own code: a run-time test cost merge 1 at 131072 x
// 2048 246 -> 262 us).
template <typename T, int Q, bool kPre, bool kSum>
__global__ void __launch_bounds__(kMThreads, 2) merge_tile_kernel(MergeArgs a, MergeGeom g) {
  extern __shared__ __align__(128) unsigned char smem[];
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem);
  uint64_t* empty_bar = full_bar + kMStages;
  float* wq = reinterpret_cast<float*>(smem + g.wq_off);
  float* gq = wq + a.d;                                      // kPre: gamma_pre
  float* red = reinterpret_cast<float*>(smem + g.red_off);  // [kMNW][3]
  float* red2 = red + kMNW * 3;                              // [kMNW] pre-norm partial sums
  unsigned char* stages = smem + g.stage_off;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int d = a.d, TM = g.TM;
  const uint32_t row_t = static_cast<uint32_t>(d) * sizeof(T);
  const uint32_t row_p = static_cast<uint32_t>(d) * 4u;
  const int np = a.nparts;
  constexpr int nx = kSum ? 1 : 0;  // the part after the running sum's, for the summary
  const bool with_p = a.P != nullptr;
  // Stage layout: O rows, then each part's rows (the summary's extra part
  // last), then P rows.
  const uint32_t p_off = static_cast<uint32_t>(TM) * row_t * static_cast<uint32_t>(1 + np + nx);
  const uint32_t tx_row = row_t * static_cast<uint32_t>(1 + np + nx) + (with_p ? row_p : 0u);
  const int64_t ntok = a.T;
  const int64_t r0 = static_cast<int64_t>(blockIdx.x) * ntok / gridDim.x;
  const int64_t r1 = static_cast<int64_t>(blockIdx.x + 1) * ntok / gridDim.x;
  const int R = static_cast<int>(r1 - r0);
  const int ntiles = (R + TM - 1) / TM;

  if (threadIdx.x == 0) {
    for (int s = 0; s < g.nst; ++s) {
      mbar_init(smem_u32(&full_bar[s]), 1);
      mbar_init(smem_u32(&empty_bar[s]), kMNW);
    }
    mbar_fence_init();
  }
  __syncthreads();

  if (warp == kMNW) {
    // ------------------------------------------------------------ producer
    if (lane != 0) return;
    int s = 0;
    uint32_t phase = 0;
    int issued = 0;
    bool ok = true;
    // O_j rows and the parts' rows of tile t into stage st.
    auto load_o = [&](unsigned char* st, int64_t row0, uint32_t rows, uint32_t fb) {
      bulk_g2s(smem_u32(st), static_cast<const T*>(a.O) + row0 * d, rows * row_t, fb);
    };
    auto load_parts = [&](unsigned char* st, int64_t row0, uint32_t rows, uint32_t fb) {
      for (int u = 0; u < np + nx; ++u)
        bulk_g2s(smem_u32(st + static_cast<uint32_t>(1 + u) * TM * row_t),
                 static_cast<const T*>(a.parts) + u * a.part_stride + row0 * d, rows * row_t, fb);
    };
    auto load_inputs = [&](unsigned char* st, int64_t row0, uint32_t rows, uint32_t fb) {
      load_o(st, row0, rows, fb);
      load_parts(st, row0, rows, fb);
    };
    // With a.early the first stages' rows that no kernel still running writes
    // are fetched before the previous kernel has finished: the parts, and
    // O_j unless a.early == 2 (the kernel before is the stage 1 that writes
    // it); O_j then and the P rows, which it may write, after.
    const int nst = g.nst;
    const int t_pre = a.early ? min(nst, ntiles) : 0;
    for (int t = 0; t < t_pre; ++t) {
      const int64_t row0 = r0 + static_cast<int64_t>(t) * R / ntiles;
      const uint32_t rows = static_cast<uint32_t>(r0 + static_cast<int64_t>(t + 1) * R / ntiles - row0);
      unsigned char* st = stages + static_cast<size_t>(t) * g.stage_bytes;
      const uint32_t fb = smem_u32(&full_bar[t]);
      mbar_arrive_expect_tx(fb, rows * tx_row);
      if (a.early == 2)
        load_parts(st, row0, rows, fb);
      else
        load_inputs(st, row0, rows, fb);
    }
    pdl_wait();
    pdl_trigger();
    for (int t = 0; t < t_pre; ++t) {
      const int64_t row0 = r0 + static_cast<int64_t>(t) * R / ntiles;
      const uint32_t rows = static_cast<uint32_t>(r0 + static_cast<int64_t>(t + 1) * R / ntiles - row0);
      unsigned char* st = stages + static_cast<size_t>(t) * g.stage_bytes;
      if (a.early == 2) load_o(st, row0, rows, smem_u32(&full_bar[t]));
      if (with_p) bulk_g2s(smem_u32(st + p_off), a.P + row0 * d, rows * row_p, smem_u32(&full_bar[t]));
    }
    issued = t_pre;
    s = t_pre % nst;
    phase = t_pre == nst ? 1u : 0u;
    for (int t = t_pre; t < ntiles; ++t) {
      if (!mbar_wait(smem_u32(&empty_bar[s]), phase ^ 1u)) {
        ok = false;
        break;
      }
      const int64_t row0 = r0 + static_cast<int64_t>(t) * R / ntiles;
      const uint32_t rows = static_cast<uint32_t>(r0 + static_cast<int64_t>(t + 1) * R / ntiles - row0);
      unsigned char* st = stages + static_cast<size_t>(s) * g.stage_bytes;
      const uint32_t fb = smem_u32(&full_bar[s]);
      if (t != a.withhold) {  // the test hook leaves this stage unfilled
        mbar_arrive_expect_tx(fb, rows * tx_row);
        load_inputs(st, row0, rows, fb);
        if (with_p) bulk_g2s(smem_u32(st + p_off), a.P + row0 * d, rows * row_p, fb);
      }
      ++issued;
      if (++s == nst) {
        s = 0;
        phase ^= 1u;
      }
    }
    if (!ok) {
      atomicOr(&g_merge_timeout, 1u);
      // Let the copies still in flight land (a withheld tile was never issued).
      for (int it = issued > nst ? issued - nst : 0; it < issued; ++it)
        if (it != a.withhold)
          (void)mbar_wait(smem_u32(&full_bar[it % nst]), static_cast<uint32_t>((it / nst) & 1));
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  // Everything below may read what the previous kernel wrote, and the next
  // kernel may start once every CTA is past this point.
  pdl_wait();
  pdl_trigger();
  for (int i = threadIdx.x; i < d; i += kMNW * 32) {
    wq[i] = a.w[i] * a.gamma[i];
    if constexpr (kPre) gq[i] = a.pre.gamma[i];
  }
  named_sync(1, kMNW * 32);
  const int wpr = g.wpr;
  const int rslot = warp / wpr;                     // row of the tile
  const int part = warp - rslot * wpr;              // part of the row
  const int span = (d + wpr - 1) / wpr;             // features per part
  const int kbeg = part * span;
  const int kend = min(d, kbeg + span);
  const float inv_d = 1.0f / static_cast<float>(d);
  int s = 0;
  uint32_t phase = 0;
  bool ok = true;
  for (int t = 0; t < ntiles; ++t) {
    const int64_t row0 = r0 + static_cast<int64_t>(t) * R / ntiles;
    const int rows = static_cast<int>(r0 + static_cast<int64_t>(t + 1) * R / ntiles - row0);
    const bool live = rslot < rows;
    const int64_t row = row0 + rslot;
    const float lse = live ? a.lse[row] : 0.f;
    // A wait that runs out is first decided per warp; the warps of a row
    // publish their outcome with their sums, so that they stop together after
    // this tile and none is left waiting at the row's named barrier.
    const bool wok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&full_bar[s]), phase));
    const unsigned char* st = stages + static_cast<size_t>(s) * g.stage_bytes;
    const T* so = reinterpret_cast<const T*>(st) + rslot * d;
    const float* sp = reinterpret_cast<const float*>(st + p_off) + rslot * d;
    // The block summary: the running sum plus the extra part, in fp32, then
    // rounded once (the freeze's sum, in its order).
    auto store_summary = [&](int k, const float (&pk)[4]) {
      float f[4];
      lds4(reinterpret_cast<const T*>(st + static_cast<uint32_t>(1 + np) * TM * row_t) + rslot * d + k, f);
      const float b4[4] = {pk[0] + f[0], pk[1] + f[1], pk[2] + f[2], pk[3] + f[3]};
      st4(static_cast<T*>(a.summary) + row * d + k, b4);
    };
    float p[Q][4];
    float ss = 0.f, dot = 0.f;
    if (Q >= 8 && wok && live) {
      // Eight chunks a lane (1024 features a warp): one pass per chunk,
      // measured faster at this width than the form below (and the form
      // below faster with four chunks or fewer).
#pragma unroll
      for (int q = 0; q < Q; ++q) {
        const int k = kbeg + (q * 32 + lane) * 4;
        if (k < kend) {
          // The running sum: the stored base (or the first part as is), then
          // the parts in order, each added in fp32.
          int u0 = 0;
          if (with_p) {
            lds4(sp + k, p[q]);
          } else {
            lds4(reinterpret_cast<const T*>(st + TM * row_t) + rslot * d + k, p[q]);
            u0 = 1;
          }
          for (int u = u0; u < np; ++u) {
            float f[4];
            lds4(reinterpret_cast<const T*>(st + static_cast<uint32_t>(1 + u) * TM * row_t) + rslot * d + k, f);
            p[q][0] += f[0]; p[q][1] += f[1]; p[q][2] += f[2]; p[q][3] += f[3];
          }
          if (a.P_out) st4(a.P_out + row * d + k, p[q]);
          if constexpr (kSum) store_summary(k, p[q]);
          const float4 w4 = *reinterpret_cast<const float4*>(wq + k);
          ss = fmaf(p[q][0], p[q][0], ss); ss = fmaf(p[q][1], p[q][1], ss);
          ss = fmaf(p[q][2], p[q][2], ss); ss = fmaf(p[q][3], p[q][3], ss);
          dot = fmaf(w4.x, p[q][0], dot); dot = fmaf(w4.y, p[q][1], dot);
          dot = fmaf(w4.z, p[q][2], dot); dot = fmaf(w4.w, p[q][3], dot);
        }
      }
    }
    if (Q < 8 && wok && live) {
      // The running sum: the stored base (or the first part as is), then the
      // parts in order, each added in fp32. One source row at a time over all
      // of the lane's chunks, so that a row's loads issue together.
      const T* part0 = reinterpret_cast<const T*>(st + TM * row_t) + rslot * d;
#pragma unroll
      for (int q = 0; q < Q; ++q) {
        const int k = kbeg + (q * 32 + lane) * 4;
        if (k < kend) {
          if (with_p)
            lds4(sp + k, p[q]);
          else
            lds4(part0 + k, p[q]);
        }
      }
      for (int u = with_p ? 0 : 1; u < np; ++u) {
        const T* fu = reinterpret_cast<const T*>(st + static_cast<uint32_t>(1 + u) * TM * row_t) + rslot * d;
#pragma unroll
        for (int q = 0; q < Q; ++q) {
          const int k = kbeg + (q * 32 + lane) * 4;
          if (k < kend) {
            float f[4];
            lds4(fu + k, f);
            p[q][0] += f[0]; p[q][1] += f[1]; p[q][2] += f[2]; p[q][3] += f[3];
          }
        }
      }
      float ss1 = 0.f, dot1 = 0.f;  // two chains each
#pragma unroll
      for (int q = 0; q < Q; ++q) {
        const int k = kbeg + (q * 32 + lane) * 4;
        if (k < kend) {
          if (a.P_out) st4(a.P_out + row * d + k, p[q]);
          if constexpr (kSum) store_summary(k, p[q]);
          const float4 w4 = *reinterpret_cast<const float4*>(wq + k);
          ss = fmaf(p[q][0], p[q][0], ss); ss1 = fmaf(p[q][1], p[q][1], ss1);
          ss = fmaf(p[q][2], p[q][2], ss); ss1 = fmaf(p[q][3], p[q][3], ss1);
          dot = fmaf(w4.x, p[q][0], dot); dot1 = fmaf(w4.y, p[q][1], dot1);
          dot = fmaf(w4.z, p[q][2], dot); dot1 = fmaf(w4.w, p[q][3], dot1);
        }
      }
      ss += ss1;
      dot += dot1;
    }
    ss = warp_sum(ss);
    dot = warp_sum(dot);
    bool rok = wok;
    if (wpr > 1) {
      if (lane == 0) {
        red[warp * 3] = ss;
        red[warp * 3 + 1] = dot;
        red[warp * 3 + 2] = wok ? 1.f : 0.f;
      }
      named_sync(2 + rslot, wpr * 32);   // only the warps of this row
      ss = 0.f;
      dot = 0.f;
      if constexpr (Q >= 8) {
        for (int w = 0; w < wpr; ++w) {
          ss += red[(rslot * wpr + w) * 3];
          dot += red[(rslot * wpr + w) * 3 + 1];
          rok = rok && red[(rslot * wpr + w) * 3 + 2] != 0.f;
        }
      } else {
#pragma unroll
        for (int w = 0; w < kMNW; ++w) {
          if (w < wpr) {
            ss += red[(rslot * wpr + w) * 3];
            dot += red[(rslot * wpr + w) * 3 + 1];
            rok = rok && red[(rslot * wpr + w) * 3 + 2] != 0.f;
          }
        }
      }
    }
    float zq = 0.f;  // this lane's share of sum(out^2), for the pre-norm
    if (rok && live) {
      const float sP = dot * rsqrtf(ss * inv_d + a.eps);
      const float M = fmaxf(lse, sP);
      const float ea = __expf(lse - M), eb = __expf(sP - M);
      const float inv = 1.0f / (ea + eb);
      const float ca = ea * inv, cb = eb * inv;
#pragma unroll
      for (int q = 0; q < Q; ++q) {
        const int k = kbeg + (q * 32 + lane) * 4;
        if (k < kend) {
          float x[4];
          lds4(so + k, x);
          // The merged row overwrites p (no longer needed).
          p[q][0] = fmaf(ca, x[0], cb * p[q][0]);
          p[q][1] = fmaf(ca, x[1], cb * p[q][1]);
          p[q][2] = fmaf(ca, x[2], cb * p[q][2]);
          p[q][3] = fmaf(ca, x[3], cb * p[q][3]);
          if (!kPre || a.out) st4(static_cast<T*>(a.out) + row * d + k, p[q]);
          zq = fmaf(p[q][0], p[q][0], zq); zq = fmaf(p[q][1], p[q][1], zq);
          zq = fmaf(p[q][2], p[q][2], zq); zq = fmaf(p[q][3], p[q][3], zq);
        }
      }
    }
    if constexpr (kPre) {
      // The sublayer's pre-norm of the merged row (its parts meet like the
      // score sums; red2 is rewritten only after the barrier below).
      zq = warp_sum(zq);
      if (wpr > 1) {
        if (lane == 0) red2[warp] = zq;
        named_sync(2 + rslot, wpr * 32);
        zq = 0.f;
        for (int w = 0; w < wpr; ++w) zq += red2[rslot * wpr + w];
      }
      if (rok && live) {
        const float rr = rsqrtf(zq * inv_d + a.pre.eps);
#pragma unroll
        for (int q = 0; q < Q; ++q) {
          const int k = kbeg + (q * 32 + lane) * 4;
          if (k < kend) {
            const float4 g4 = *reinterpret_cast<const float4*>(gq + k);
            const float y[4] = {g4.x * (p[q][0] * rr), g4.y * (p[q][1] * rr), g4.z * (p[q][2] * rr),
                                g4.w * (p[q][3] * rr)};
            st4(static_cast<T*>(a.pre.out) + row * d + k, y);
          }
        }
      }
    }
    if (wpr > 1) named_sync(2 + rslot, wpr * 32);  // partners are done reading red[] and red2[]
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&empty_bar[s]));
    if (++s == g.nst) {
      s = 0;
      phase ^= 1u;
    }
    if (!rok) {
      ok = false;
      break;
    }
  }
  if (!ok && lane == 0) atomicOr(&g_merge_timeout, 1u);
}

// ---------------------------------------------------------- general merge --

// The running sum of one element: the stored base (or the first part as is),
// then the parts in order, each added in fp32.
template <typename T>
__device__ __forceinline__ float running_sum_at(const float* P, const void* parts, int64_t part_stride, int np,
                                                int64_t off) {
  const T* f = static_cast<const T*>(parts);
  float p;
  int u = 0;
  if (P) {
    p = P[off];
  } else {
    p = to_f32(f[off]);
    u = 1;
  }
  for (; u < np; ++u) p += to_f32(f[u * part_stride + off]);
  return p;
}

template <typename T>
__global__ void __launch_bounds__(kBlock) merge_generic_kernel(MergeArgs a) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int d = a.d;
  const float inv_d = 1.0f / static_cast<float>(d);
  // Each lane forms and writes only the elements it owns, so P_out may be P;
  // with no P_out the running sum is formed again where it is needed.
  for (int64_t row = static_cast<int64_t>(blockIdx.x) * kWarps + warp; row < a.T;
       row += static_cast<int64_t>(gridDim.x) * kWarps) {
    float ss = 0.f, dot = 0.f;
    for (int k = lane; k < d; k += 32) {
      const int64_t off = row * d + k;
      const float p = running_sum_at<T>(a.P, a.parts, a.part_stride, a.nparts, off);
      if (a.P_out) a.P_out[off] = p;
      if (a.summary)  // the block summary: one part more, then rounded
        static_cast<T*>(a.summary)[off] =
            from_f32<T>(p + to_f32(static_cast<const T*>(a.parts)[a.nparts * a.part_stride + off]));
      ss = fmaf(p, p, ss);
      dot = fmaf(a.w[k] * a.gamma[k], p, dot);
    }
    ss = warp_sum(ss);
    dot = warp_sum(dot);
    const float s = dot * rsqrtf(ss * inv_d + a.eps);
    const float lse = a.lse[row];  // general path: simplicity over latency
    const float M = fmaxf(lse, s);
    const float ea = __expf(lse - M), eb = __expf(s - M);
    const float inv = 1.0f / (ea + eb);
    // The running sum again: from P_out where it was stored (P may be P_out).
    const float* Pn = a.P_out;
    float zq = 0.f;
    for (int k = lane; k < d; k += 32) {
      const int64_t off = row * d + k;
      const float o = to_f32(static_cast<const T*>(a.O)[off]);
      const float p = Pn ? Pn[off] : running_sum_at<T>(a.P, a.parts, a.part_stride, a.nparts, off);
      const float z = fmaf(ea * inv, o, eb * inv * p);
      if (a.out) static_cast<T*>(a.out)[off] = from_f32<T>(z);
      zq = fmaf(z, z, zq);
    }
    if (a.pre.gamma) {
      // The sublayer's pre-norm: the merged row again, scaled by 1 / its rms.
      const float rr = rsqrtf(warp_sum(zq) * inv_d + a.pre.eps);
      for (int k = lane; k < d; k += 32) {
        const int64_t off = row * d + k;
        const float o = to_f32(static_cast<const T*>(a.O)[off]);
        const float p = Pn ? Pn[off] : running_sum_at<T>(a.P, a.parts, a.part_stride, a.nparts, off);
        const float z = fmaf(ea * inv, o, eb * inv * p);
        static_cast<T*>(a.pre.out)[off] = from_f32<T>(a.pre.gamma[k] * (z * rr));
      }
    }
  }
}

// ------------------------------------------------------------- RMSNorm ------
// out = gamma * x / sqrt(mean(x^2) + eps) per row, one warp per row, fp32
// arithmetic; the sublayer pre-norm of a row that needs no merge (the first
// sublayer of a block, whose output stage 1 writes).
template <typename T>
__global__ void __launch_bounds__(kBlock) rmsnorm_kernel(const T* x, int64_t ntok, int d, const float* gamma,
                                                        float eps, T* out) {
  pdl_trigger();
  pdl_wait();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const float inv_d = 1.0f / static_cast<float>(d);
  for (int64_t row = static_cast<int64_t>(blockIdx.x) * kWarps + warp; row < ntok;
       row += static_cast<int64_t>(gridDim.x) * kWarps) {
    const T* xr = x + row * d;
    float q = 0.f;
    for (int k = lane; k < d; k += 32) {
      const float v = to_f32(xr[k]);
      q = fmaf(v, v, q);
    }
    const float rr = rsqrtf(warp_sum(q) * inv_d + eps);
    // Each lane rewrites only the elements it read, so out may be x.
    for (int k = lane; k < d; k += 32) out[row * d + k] = from_f32<T>(gamma[k] * (to_f32(xr[k]) * rr));
  }
}

// ------------------------------------------------------- accumulate/freeze --

template <typename T>
__global__ void __launch_bounds__(kBlock) accum_fast_kernel(AccumArgs a, int64_t nchunks) {
  pdl_trigger();
  if (!a.no_wait) pdl_wait();
  const T* f = static_cast<const T*>(a.parts);
  for (int64_t c = static_cast<int64_t>(blockIdx.x) * kBlock + threadIdx.x; c < nchunks;
       c += static_cast<int64_t>(gridDim.x) * kBlock) {
    const int64_t off = c * 4;
    float p[4];
    int u = 0;
    if (a.P) {
      ldg4(a.P + off, p);
    } else {
      ldg4(f + off, p);
      u = 1;
    }
    for (; u < a.nparts; ++u) {
      float x[4];
      ldg4(f + u * a.part_stride + off, x);
      p[0] += x[0]; p[1] += x[1]; p[2] += x[2]; p[3] += x[3];
    }
    if (a.summary)
      st4(static_cast<T*>(a.summary) + off, p);
    else
      st4(a.P_out + off, p);
  }
}

template <typename T>
__global__ void __launch_bounds__(kBlock) accum_generic_kernel(AccumArgs a, int64_t n) {
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * kBlock + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * kBlock) {
    const float p = running_sum_at<T>(a.P, a.parts, a.part_stride, a.nparts, i);
    if (a.summary)
      static_cast<T*>(a.summary)[i] = from_f32<T>(p);
    else
      a.P_out[i] = p;
  }
}

// Enough blocks for the work, at most one resident wave of `kernel`.
unsigned grid_for(int64_t work_items, int per_block, const void* kernel) {
  int64_t blocks = (work_items + per_block - 1) / per_block;
  const int64_t cap = static_cast<int64_t>(sm_count()) * blocks_per_sm(kernel, kBlock, 0);
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  return static_cast<unsigned>(blocks);
}

}  // namespace

bool merge_fast_ok(const MergeArgs& a) {
  const int es = a.bf16 ? 2 : 4;
  if (a.d % 4 != 0 || (a.d * es) % 16 != 0) return false;
  if ((a.part_stride * es) % 16 != 0) return false;
  const int nx = a.summary ? 1 : 0;
  const MergeGeom g = merge_geom(a.d, es, a.pre.gamma != nullptr, a.nparts + nx, a.P != nullptr);
  const int per_warp = (a.d + g.wpr - 1) / g.wpr;
  // Every part of a row starts on a 4-feature chunk (aligned vector loads).
  if (per_warp % 4 != 0 || per_warp > 8 * 128 || g.total > 227 * 1024) return false;
  return aligned16(a.O) && aligned16(a.P) && aligned16(a.P_out) && aligned16(a.out) && aligned16(a.summary) &&
         (a.nparts + nx == 0 || aligned16(a.parts)) &&
         (!a.pre.gamma || (aligned16(a.pre.gamma) && aligned16(a.pre.out)));
}

bool accum_fast_ok(const AccumArgs& a) {
  const int es = a.bf16 ? 2 : 4;
  if (a.d % 4 != 0 || (a.part_stride * es) % 16 != 0) return false;
  return aligned16(a.P) && aligned16(a.P_out) && aligned16(a.parts) && aligned16(a.summary);
}

namespace {
template <typename T, int Q>
cudaError_t launch_merge_tiles(const MergeArgs& a, const MergeGeom& g, cudaStream_t s) {
  auto k = a.pre.gamma ? merge_tile_kernel<T, Q, true, false>
                       : (a.summary ? merge_tile_kernel<T, Q, false, true> : merge_tile_kernel<T, Q, false, false>);
  cudaError_t e = allow_dynamic_smem(reinterpret_cast<const void*>(k), g.total);
  if (e != cudaSuccess) return e;
  int64_t grid = (a.T + g.TM - 1) / g.TM;
  const int64_t cap = static_cast<int64_t>(sm_count()) * blocks_per_sm(reinterpret_cast<const void*>(k), kMThreads, g.total);
  if (grid > cap) grid = cap;
  return launch_pdl(k, static_cast<unsigned>(grid), kMThreads, g.total, s, a, g);
}

template <typename T>
cudaError_t launch_merge_dtype(const MergeArgs& a, cudaStream_t s) {
  const MergeGeom g = merge_geom(a.d, sizeof(T), a.pre.gamma != nullptr, a.nparts + (a.summary ? 1 : 0),
                                 a.P != nullptr);
  const int per_warp = (a.d + g.wpr - 1) / g.wpr;
  int q = 1;
  while (q * 128 < per_warp) q <<= 1;
  switch (q) {
    case 1: return launch_merge_tiles<T, 1>(a, g, s);
    case 2: return launch_merge_tiles<T, 2>(a, g, s);
    case 4: return launch_merge_tiles<T, 4>(a, g, s);
    case 8: return launch_merge_tiles<T, 8>(a, g, s);
    default: return cudaErrorInvalidValue;
  }
}
}  // namespace

cudaError_t take_timeout_merge(unsigned int* flag) {
  unsigned int zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(flag, g_merge_timeout, sizeof(unsigned int));
  if (e != cudaSuccess) return e;
  return cudaMemcpyToSymbol(g_merge_timeout, &zero, sizeof(unsigned int));
}

cudaError_t launch_merge(const MergeArgs& a, cudaStream_t s, bool fast) {
  if (fast) return a.bf16 ? launch_merge_dtype<bf16>(a, s) : launch_merge_dtype<float>(a, s);
  if (a.bf16) {
    auto k = merge_generic_kernel<bf16>;
    k<<<grid_for(a.T, kWarps, reinterpret_cast<const void*>(k)), kBlock, 0, s>>>(a);
  } else {
    auto k = merge_generic_kernel<float>;
    k<<<grid_for(a.T, kWarps, reinterpret_cast<const void*>(k)), kBlock, 0, s>>>(a);
  }
  return cudaGetLastError();
}

cudaError_t launch_rmsnorm(const void* x, int64_t T, int d, int is_bf16, const float* gamma, float eps, void* out,
                           cudaStream_t s) {
  const int64_t blocks = (T + kWarps - 1) / kWarps;
  if (is_bf16) {
    auto k = rmsnorm_kernel<bf16>;
    return launch_pdl(k, grid_for(blocks * kBlock, kBlock, reinterpret_cast<const void*>(k)), kBlock, 0, s,
                      static_cast<const bf16*>(x), T, d, gamma, eps, static_cast<bf16*>(out));
  }
  auto k = rmsnorm_kernel<float>;
  return launch_pdl(k, grid_for(blocks * kBlock, kBlock, reinterpret_cast<const void*>(k)), kBlock, 0, s,
                    static_cast<const float*>(x), T, d, gamma, eps, static_cast<float*>(out));
}

cudaError_t launch_accum(const AccumArgs& a, cudaStream_t s, bool fast) {
  const int64_t total = a.T * a.d;
  if (fast) {
    const int64_t nchunks = total / 4;
    if (a.bf16) {
      auto k = accum_fast_kernel<bf16>;
      return launch_pdl(k, grid_for(nchunks, kBlock, reinterpret_cast<const void*>(k)), kBlock, 0, s, a, nchunks);
    }
    auto k = accum_fast_kernel<float>;
    return launch_pdl(k, grid_for(nchunks, kBlock, reinterpret_cast<const void*>(k)), kBlock, 0, s, a, nchunks);
  }
  if (a.bf16) {
    auto k = accum_generic_kernel<bf16>;
    k<<<grid_for(total, kBlock, reinterpret_cast<const void*>(k)), kBlock, 0, s>>>(a, total);
  } else {
    auto k = accum_generic_kernel<float>;
    k<<<grid_for(total, kBlock, reinterpret_cast<const void*>(k)), kBlock, 0, s>>>(a, total);
  }
  return cudaGetLastError();
}

}  // namespace attnres
