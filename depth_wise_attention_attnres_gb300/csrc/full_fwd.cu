// Full AttnRes read, fast kernel (sm_103a).
//
// Computes, per token row t (DepthBench reading notes section 2.3, paper
// Appendix A; LLMRes blog "Kimi AttnRes"):
//   e_i = w^T (gamma * v_i / sqrt(mean(v_i^2) + eps)),  z = sum_i softmax_i(e) v_i
// in one pass over the sources with an online softmax (running max m and mass
// l; the accumulator is rescaled only when the max grows).
//
// Data movement: each CTA owns a contiguous range of token rows and walks it
// in tiles of kTM rows. For every (tile, source) pair the rows are contiguous
// in HBM ([n, T, d] layout), so one elected producer thread moves the whole
// tile with a single 1-D bulk copy (cp.async.bulk, TMA engine) into a ring of
// shared-memory stages guarded by mbarriers. Eight consumer warps each own
// one row of the tile: a lane holds d/32 elements (4 consecutive per 128-element
// chunk, conflict-free 8/16-byte shared loads), the RMS and the score are two
// butterfly warp sums, and the weighted accumulation stays in fp32 registers.
// The path is HBM-bound (one pass, about 3 flop per byte), so tensor cores are
// not used.
#include <math.h>

#include "common.cuh"
#include "internal.h"

namespace attnres {
namespace {

__device__ unsigned int g_full_timeout = 0;

constexpr int kBarBytes = 128;       // barrier area at the start of shared memory
constexpr int kMaxStages = 8;
constexpr int kSmemPerSM = 224 * 1024;  // shared memory the CTAs of one SM split

// Rows up to 1024 wide run two CTAs per SM (16 consumer warps hide the
// latency of the per-source reduction chain); that caps registers at 112.
// Per row width (CH = d / 128): NW consumer warps per CTA (= rows per tile)
// and CTAs per SM. Several CTAs per SM run independent pipelines, so their
// warps do not all wait and reduce in lockstep; the register budget (all
// CTAs' threads share 64K registers) decides how many fit.
template <int CH>
struct FullTraits {
  static constexpr int kNW = 8;
  static constexpr int kMinBlocks = CH <= 5 ? 3 : (CH <= 8 ? 2 : 1);
  // Keeping the converted row in registers saves a second shared read when
  // the registers allow it.
  static constexpr bool kKeepX = CH <= 4 || (CH >= 6 && CH <= 8);
  // fp32 values in shared memory before the stages: w * gamma, plus gamma_pre
  // (mode 1) or one query row per consumer warp (mode 2).
  static constexpr int fixed_floats(int mode) { return CH * 128 * (mode == 1 ? 2 : (mode == 2 ? 1 + kNW : 1)); }
};

// kMode 0: the read; 1: the epilogue also writes the sublayer pre-norm of the
// row; 2: every token has its own query (a.Q, the input-dependent query),
// staged per row in shared memory. Separate instances, so the plain read
// keeps its own code and schedule.
template <typename Tin, int CH, int kMode>
__global__ void __launch_bounds__((FullTraits<CH>::kNW + 1) * kWarp, FullTraits<CH>::kMinBlocks)
    full_fwd_bulk_kernel(FullArgs a, int nstage) {
  constexpr int kNW = FullTraits<CH>::kNW;  // consumer warps = rows per tile
  constexpr int kTM = kNW;
  constexpr int D = CH * 128;
  constexpr int NE = CH * 4;         // elements per lane
  constexpr bool kKeepX = FullTraits<CH>::kKeepX;

  extern __shared__ __align__(128) unsigned char smem[];
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem);
  uint64_t* empty_bar = full_bar + kMaxStages;
  float* wq = reinterpret_cast<float*>(smem + kBarBytes);  // w * gamma, [D]
  constexpr bool kPre = kMode == 1, kDynQ = kMode == 2;
  float* gq = wq + D;                                       // kPre: gamma_pre, [D]; kDynQ: q * gamma rows [kNW][D]
  Tin* stages = reinterpret_cast<Tin*>(smem + kBarBytes + FullTraits<CH>::fixed_floats(kMode) * sizeof(float));
  constexpr int kStageElems = kTM * D;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int64_t T = a.T;
  // Contiguous rows [r0, r1) per CTA, cut into ntiles tiles whose sizes
  // differ by at most one row (tile t starts at r0 + t * R / ntiles).
  const int64_t r0 = static_cast<int64_t>(blockIdx.x) * T / gridDim.x;
  const int64_t r1 = static_cast<int64_t>(blockIdx.x + 1) * T / gridDim.x;
  const int R = static_cast<int>(r1 - r0);
  const int ntiles = (R + kTM - 1) / kTM;
  const int n = a.n_src;
  const int64_t total = static_cast<int64_t>(ntiles) * n;

  // A read that waits for the previous kernel at its start lets the next one
  // launch only after that wait: a later read of the same pass (which does not
  // wait at its start) then never runs ahead of whatever wrote the sources.
  if (a.late_wait) pdl_trigger();
  if (threadIdx.x == 0) {
    for (int s = 0; s < nstage; ++s) {
      mbar_init(smem_u32(&full_bar[s]), 1);
      mbar_init(smem_u32(&empty_bar[s]), kNW);
    }
    mbar_fence_init();
  }
  __syncthreads();
  // Everything below may read what the previous kernel wrote, unless this is
  // a later read of a pass, whose inputs the previous read does not write (it
  // then waits before it ends, so reads still complete in order).
  if (!a.late_wait) {
    pdl_wait();
    pdl_trigger();
  }

  if (warp == kNW) {
    // ------------------------------------------------------------ producer
    if (lane != 0) return;
    const char* V = static_cast<const char*>(a.V);
    int stage = 0;
    uint32_t phase = 0;
    int64_t issued = 0;
    bool ok = true;
    for (int64_t it = 0; it < total; ++it) {
      // A fresh barrier counts its (virtual) previous phase as complete, so
      // the first round of waits on parity 1 passes at once.
      if (!mbar_wait(smem_u32(&empty_bar[stage]), phase ^ 1u)) {
        ok = false;
        break;
      }
      const int tile = static_cast<int>(it / n);
      const int src = static_cast<int>(it - static_cast<int64_t>(tile) * n);
      const int64_t row0 = r0 + tile * R / ntiles;
      const int rows = static_cast<int>(r0 + (tile + 1) * R / ntiles - row0);
      const uint32_t bytes = static_cast<uint32_t>(rows) * D * sizeof(Tin);
      const uint32_t fb = smem_u32(&full_bar[stage]);
      if (it != a.withhold) {  // the test hook leaves this stage unfilled
        mbar_arrive_expect_tx(fb, bytes);
        bulk_g2s(smem_u32(stages + static_cast<size_t>(stage) * kStageElems),
                 V + (static_cast<int64_t>(src) * a.src_stride + row0 * D) * sizeof(Tin), bytes, fb);
      }
      ++issued;
      if (++stage == nstage) {
        stage = 0;
        phase ^= 1u;
      }
    }
    if (!ok) {
      atomicOr(&g_full_timeout, 1u);
      // Let the copies still in flight land before this CTA's memory goes
      // (a withheld copy was never issued).
      for (int64_t it = issued > nstage ? issued - nstage : 0; it < issued; ++it)
        if (it != a.withhold)
          (void)mbar_wait(smem_u32(&full_bar[it % nstage]), static_cast<uint32_t>((it / nstage) & 1));
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  // w * gamma into shared memory; the producer is already streaming meanwhile.
  for (int i = threadIdx.x; i < D / 4; i += kNW * kWarp) {
    if constexpr (!kDynQ) {  // with per-token queries there is no shared w
      const float4 w4 = reinterpret_cast<const float4*>(a.w)[i];
      const float4 g4 = reinterpret_cast<const float4*>(a.gamma)[i];
      reinterpret_cast<float4*>(wq)[i] = make_float4(w4.x * g4.x, w4.y * g4.y, w4.z * g4.z, w4.w * g4.w);
    }
    if constexpr (kPre) reinterpret_cast<float4*>(gq)[i] = reinterpret_cast<const float4*>(a.pre.gamma)[i];
  }
  named_sync(1, kNW * kWarp);
  const float inv_d = 1.0f / static_cast<float>(D);
  const float eps = a.eps;

  int stage = 0;
  uint32_t phase = 0;
  bool ok = true;
  for (int tile = 0; tile < ntiles && ok; ++tile) {
    const int64_t row0 = r0 + tile * R / ntiles;
    const int64_t row = row0 + warp;
    const bool valid = row < r0 + (tile + 1) * R / ntiles;
    float2 acc[NE / 2];
#pragma unroll
    for (int e = 0; e < NE / 2; ++e) acc[e] = make_float2(0.f, 0.f);
    float m = -INFINITY, l = 0.f;
    const float* qrow = wq;  // the query (times gamma) this row is scored with
    if constexpr (kDynQ) {
      float* qr = gq + warp * D;
      if (valid) {
#pragma unroll
        for (int c = 0; c < CH; ++c) {
          const int k = (c * kWarp + lane) * 4;
          const float4 q4 = *reinterpret_cast<const float4*>(a.Q + row * D + k);
          const float4 g4 = *reinterpret_cast<const float4*>(a.gamma + k);
          *reinterpret_cast<float4*>(qr + k) = make_float4(q4.x * g4.x, q4.y * g4.y, q4.z * g4.z, q4.w * g4.w);
        }
      }
      __syncwarp();
      qrow = qr;
    }

    for (int src = 0; src < n; ++src) {
      if (!mbar_wait(smem_u32(&full_bar[stage]), phase)) {
        ok = false;
        break;
      }
      if (valid) {
        const Tin* rowp = stages + static_cast<size_t>(stage) * kStageElems + warp * D;
        float x[kKeepX ? NE : 4];
        float2 ss2a = make_float2(0.f, 0.f), ss2b = ss2a, dt2a = ss2a, dt2b = ss2a;
#pragma unroll
        for (int c = 0; c < CH; ++c) {
          float t4[4];
          lds4(rowp + (c * kWarp + lane) * 4, t4);
          if constexpr (kKeepX) {
            x[c * 4 + 0] = t4[0]; x[c * 4 + 1] = t4[1]; x[c * 4 + 2] = t4[2]; x[c * 4 + 3] = t4[3];
          }
          const float2 xa = make_float2(t4[0], t4[1]);
          const float2 xb = make_float2(t4[2], t4[3]);
          ss2a = ffma2(xa, xa, ss2a);
          ss2b = ffma2(xb, xb, ss2b);
          const float4 w4 = *reinterpret_cast<const float4*>(qrow + (c * kWarp + lane) * 4);
          dt2a = ffma2(make_float2(w4.x, w4.y), xa, dt2a);
          dt2b = ffma2(make_float2(w4.z, w4.w), xb, dt2b);
        }
        (void)x;
        const float ss = warp_sum((ss2a.x + ss2b.x) + (ss2a.y + ss2b.y));
        const float dot = warp_sum((dt2a.x + dt2b.x) + (dt2a.y + dt2b.y));
        const float s = dot * rsqrtf(ss * inv_d + eps);
        if (s > m) {  // warp-uniform: s and m are identical on every lane
          const float c = __expf(m - s);
          l *= c;
          const float2 c2 = make_float2(c, c);
#pragma unroll
          for (int e = 0; e < NE / 2; ++e) acc[e] = fmul2(acc[e], c2);
          m = s;
        }
        const float p = __expf(s - m);
        l += p;
        const float2 p2 = make_float2(p, p);
        if constexpr (kKeepX) {
#pragma unroll
          for (int e = 0; e < NE / 2; ++e) acc[e] = ffma2(p2, make_float2(x[2 * e], x[2 * e + 1]), acc[e]);
        } else {
#pragma unroll
          for (int c = 0; c < CH; ++c) {
            float t4[4];
            lds4(rowp + (c * kWarp + lane) * 4, t4);
            acc[c * 2] = ffma2(p2, make_float2(t4[0], t4[1]), acc[c * 2]);
            acc[c * 2 + 1] = ffma2(p2, make_float2(t4[2], t4[3]), acc[c * 2 + 1]);
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&empty_bar[stage]));
      if (++stage == nstage) {
        stage = 0;
        phase ^= 1u;
      }
    }

    if (!kPre && ok && valid) {
      const float inv = 1.0f / l;
#pragma unroll
      for (int c = 0; c < CH; ++c) {
        const int k = (c * kWarp + lane) * 4;
        const float o[4] = {acc[c * 2].x * inv, acc[c * 2].y * inv, acc[c * 2 + 1].x * inv,
                            acc[c * 2 + 1].y * inv};
        if (a.out_bf16)
          st4(static_cast<bf16*>(a.out) + row * D + k, o);
        else
          st4(static_cast<float*>(a.out) + row * D + k, o);
      }
    } else if (kPre && ok && valid) {
      // With the sublayer's pre-norm: z (if it is wanted), then
      // gamma_pre * z / rms(z) from z in fp32.
      const float inv = 1.0f / l;
      const float2 inv2 = make_float2(inv, inv);
#pragma unroll
      for (int e = 0; e < NE / 2; ++e) acc[e] = fmul2(acc[e], inv2);
      float2 q2 = make_float2(0.f, 0.f);
#pragma unroll
      for (int c = 0; c < CH; ++c) {
        const int k = (c * kWarp + lane) * 4;
        q2 = ffma2(acc[c * 2], acc[c * 2], q2);
        q2 = ffma2(acc[c * 2 + 1], acc[c * 2 + 1], q2);
        if (a.out) {
          const float o[4] = {acc[c * 2].x, acc[c * 2].y, acc[c * 2 + 1].x, acc[c * 2 + 1].y};
          if (a.out_bf16)
            st4(static_cast<bf16*>(a.out) + row * D + k, o);
          else
            st4(static_cast<float*>(a.out) + row * D + k, o);
        }
      }
      const float rr = rsqrtf(warp_sum(q2.x + q2.y) * inv_d + a.pre.eps);
#pragma unroll
      for (int c = 0; c < CH; ++c) {
        const int k = (c * kWarp + lane) * 4;
        const float4 g4 = *reinterpret_cast<const float4*>(gq + k);
        const float o[4] = {g4.x * (acc[c * 2].x * rr), g4.y * (acc[c * 2].y * rr), g4.z * (acc[c * 2 + 1].x * rr),
                            g4.w * (acc[c * 2 + 1].y * rr)};
        if (a.out_bf16)
          st4(static_cast<bf16*>(a.pre.out) + row * D + k, o);
        else
          st4(static_cast<float*>(a.pre.out) + row * D + k, o);
      }
    }
  }
  if (!ok) atomicOr(&g_full_timeout, 1u);
  if (a.late_wait) pdl_wait();
}

template <typename Tin, int CH, int kMode>
cudaError_t launch_chp(const FullArgs& a, cudaStream_t s) {
  constexpr int D = CH * 128;
  constexpr int kTM = FullTraits<CH>::kNW;
  constexpr int kThreads = (kTM + 1) * kWarp;
  const int stage_bytes = kTM * D * static_cast<int>(sizeof(Tin));
  const int fixed = kBarBytes + FullTraits<CH>::fixed_floats(kMode) * static_cast<int>(sizeof(float));
  int nstage = (kSmemPerSM / FullTraits<CH>::kMinBlocks - 1024 - fixed) / stage_bytes;
  nstage = nstage < 2 ? 2 : (nstage > kMaxStages ? kMaxStages : nstage);
  const int smem = fixed + nstage * stage_bytes;
  const void* fn = reinterpret_cast<const void*>(&full_fwd_bulk_kernel<Tin, CH, kMode>);
  cudaError_t e = allow_dynamic_smem(fn, smem);
  if (e != cudaSuccess) return e;
  const int per_sm = blocks_per_sm(fn, kThreads, smem);
  const int64_t tiles = (a.T + kTM - 1) / kTM;
  int64_t grid = static_cast<int64_t>(sm_count()) * (per_sm > 0 ? per_sm : 1);
  if (grid > tiles) grid = tiles;
  return launch_pdl(full_fwd_bulk_kernel<Tin, CH, kMode>, static_cast<unsigned>(grid), kThreads, smem, s, a,
                    nstage);
}

template <typename Tin, int CH>
cudaError_t launch_ch(const FullArgs& a, cudaStream_t s) {
  if (a.Q) return launch_chp<Tin, CH, 2>(a, s);
  return a.pre.gamma ? launch_chp<Tin, CH, 1>(a, s) : launch_chp<Tin, CH, 0>(a, s);
}

template <typename Tin>
cudaError_t launch_dtype(const FullArgs& a, cudaStream_t s) {
  switch (a.d / 128) {
    case 1: return launch_ch<Tin, 1>(a, s);
    case 2: return launch_ch<Tin, 2>(a, s);
    case 3: return launch_ch<Tin, 3>(a, s);
    case 4: return launch_ch<Tin, 4>(a, s);
    case 5: return launch_ch<Tin, 5>(a, s);
    case 6: return launch_ch<Tin, 6>(a, s);
    case 7: return launch_ch<Tin, 7>(a, s);
    case 8: return launch_ch<Tin, 8>(a, s);
    case 10: return launch_ch<Tin, 10>(a, s);
    case 12: return launch_ch<Tin, 12>(a, s);
    case 16: return launch_ch<Tin, 16>(a, s);
    default: return cudaErrorInvalidValue;
  }
}

// One mbarrier that nothing ever arrives on: the bounded wait must give up,
// record the timeout and let the kernel return.
__global__ void wait_timeout_selftest_kernel() {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    mbar_fence_init();
  }
  __syncthreads();
  if (!mbar_wait(smem_u32(&bar), 0u)) atomicOr(&g_full_timeout, 1u);
}

}  // namespace

cudaError_t launch_wait_timeout_selftest(cudaStream_t s) {
  wait_timeout_selftest_kernel<<<1, 32, 0, s>>>();
  return cudaGetLastError();
}

bool full_fast_ok(const FullArgs& a) {
  const int es = a.v_bf16 ? 2 : 4;
  const int ch = a.d / 128;
  const bool ch_ok = (a.d % 128 == 0) && ((ch >= 1 && ch <= 8) || ch == 10 || ch == 12 || ch == 16);
  return ch_ok && aligned16(a.V) && aligned16(a.out) && aligned16(a.w) && aligned16(a.gamma) &&
         ((a.src_stride * es) % 16 == 0) && (!a.pre.gamma || (aligned16(a.pre.gamma) && aligned16(a.pre.out))) &&
         aligned16(a.Q) && !(a.Q && a.pre.gamma);
}

cudaError_t launch_full_fast(const FullArgs& a, cudaStream_t s) {
  return a.v_bf16 ? launch_dtype<bf16>(a, s) : launch_dtype<float>(a, s);
}

cudaError_t take_timeout_full(unsigned int* flag) {
  unsigned int zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(flag, g_full_timeout, sizeof(unsigned int));
  if (e != cudaSuccess) return e;
  return cudaMemcpyToSymbol(g_full_timeout, &zero, sizeof(unsigned int));
}

}  // namespace attnres
