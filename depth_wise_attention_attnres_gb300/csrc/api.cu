// C ABI of the AttnRes aggregation library: argument checks, kernel choice,
// pass sequencing and device status. Every computation runs in the kernels of
// the other .cu files.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <atomic>
#include <map>
#include <mutex>
#include <tuple>

#include "attnres.h"
#include "internal.h"

namespace attnres {

namespace {
std::mutex g_mu;
// (kernel, context) -> dynamic shared memory bytes allowed. A kernel's
// attributes belong to a context: a device reset makes a new one, which must
// be set up again.
std::map<std::pair<const void*, unsigned long long>, int> g_smem_set;
std::map<std::tuple<const void*, int, int, int>, int> g_occ;      // (kernel, dev, thr, smem)
std::map<int, int> g_sms;

int current_device() {
  int dev = 0;
  cudaGetDevice(&dev);
  return dev;
}

// Process-unique id of the current context (cuCtxGetId), or, when there is
// none yet or the driver cannot say, the device number with the top bit set.
// Two driver queries, no synchronisation (also fine inside stream capture).
unsigned long long current_context_key() {
  static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
  static PFN_cuCtxGetId_v12000 get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(p);
    cudaGetLastError();
  });
  const unsigned long long fallback = (1ull << 63) | static_cast<unsigned long long>(current_device());
  if (!get_current || !get_id) return fallback;
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (get_current(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, &id) != CUDA_SUCCESS) return fallback;
  return id;
}
}  // namespace

int sm_count() {
  const int dev = current_device();
  std::lock_guard<std::mutex> lk(g_mu);
  auto it = g_sms.find(dev);
  if (it != g_sms.end()) return it->second;
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1) n = 1;
  g_sms[dev] = n;
  return n;
}

// Lets `kernel` use `bytes` of dynamic shared memory and asks for the largest
// shared-memory carveout, so that the CTAs the occupancy allows fit. Done
// once per (kernel, context); later calls only look the answer up.
cudaError_t allow_dynamic_smem(const void* kernel, int bytes) {
  const unsigned long long ctx = current_context_key();
  std::lock_guard<std::mutex> lk(g_mu);
  auto key = std::make_pair(kernel, ctx);
  auto it = g_smem_set.find(key);
  if (it != g_smem_set.end() && it->second >= bytes) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                       cudaSharedmemCarveoutMaxShared);
  if (e != cudaSuccess) return e;
  // Without the attribute, static and dynamic shared memory together are
  // held to 48 KB, so it is set for any dynamic size.
  if (bytes > 0) {
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return e;
  }
  g_smem_set[key] = bytes;
  return cudaSuccess;
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

int blocks_per_sm(const void* kernel, int threads, int smem_bytes) {
  const int dev = current_device();
  std::lock_guard<std::mutex> lk(g_mu);
  auto key = std::make_tuple(kernel, dev, threads, smem_bytes);
  auto it = g_occ.find(key);
  if (it != g_occ.end()) return it->second;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, threads, smem_bytes) != cudaSuccess) {
    cudaGetLastError();
    n = 1;
  }
  if (n < 1) n = 1;
  g_occ[key] = n;
  return n;
}

// Failure-path test hook (attnres_test_withhold_stage), off by default.
namespace {
std::atomic<int> g_withhold_kernel{kWithholdNone};
std::atomic<int64_t> g_withhold_index{-1};
}  // namespace

int64_t withhold_for(WithholdKernel k) {
  return g_withhold_kernel.load() == k ? g_withhold_index.load() : -1;
}

}  // namespace attnres

using namespace attnres;

namespace {

constexpr int kGenericScoreLimit = 200 * 1024;  // bytes of scores per warp

bool valid_dtype(int32_t t) { return t == ATTNRES_F32 || t == ATTNRES_BF16; }
int elem_size(int32_t t) { return t == ATTNRES_BF16 ? 2 : 4; }
bool valid_eps(float eps) { return eps >= 0.0f && eps < 3.0e38f; }

struct Range {
  uintptr_t lo = 0, hi = 0;  // [lo, hi)
};
Range range_of(const void* p, int64_t bytes) {
  Range r;
  r.lo = reinterpret_cast<uintptr_t>(p);
  r.hi = r.lo + static_cast<uintptr_t>(bytes);
  return r;
}
bool overlap(const Range& a, const Range& b) {
  if (a.lo == a.hi || b.lo == b.hi) return false;
  return a.lo < b.hi && b.lo < a.hi;
}

int status_of(cudaError_t e) {
  if (e == cudaSuccess) return ATTNRES_OK;
  cudaGetLastError();  // consume it
  return e == cudaErrorInvalidValue ? ATTNRES_ERR_UNSUPPORTED : ATTNRES_ERR_CUDA;
}

cudaStream_t as_stream(void* s) { return static_cast<cudaStream_t>(s); }

// Failure-path test hook (attnres_test_fail_launch): the launch after
// g_fail_after more successful ones reports a CUDA error without being
// made. -1, the default, injects nothing.
std::atomic<int64_t> g_fail_after{-1};

bool injected_failure() {
  int64_t v = g_fail_after.load();
  while (v >= 0) {
    if (g_fail_after.compare_exchange_weak(v, v - 1)) return v == 0;
  }
  return false;
}

// Every launch (kernel, memset or copy) the library makes goes through here:
// the test hook first, then the launch and its status.
template <typename F>
int launched(F&& launch) {
  if (injected_failure()) return ATTNRES_ERR_CUDA;
  return status_of(launch());
}

// Checks and fills the arguments of one full read. Returns a status.
int make_full(const void* V, int64_t src_stride, int32_t n_src, int64_t T, int32_t d,
              int32_t v_dtype, const float* w, const float* gamma, float eps, void* out,
              int32_t out_dtype, FullArgs* a) {
  if (n_src < 1 || d < 1 || T < 0 || !valid_dtype(v_dtype) || !valid_dtype(out_dtype) ||
      !valid_eps(eps))
    return ATTNRES_ERR_INVALID_ARG;
  if (T == 0) return ATTNRES_OK;
  if (!V || !w || !gamma || !out) return ATTNRES_ERR_INVALID_ARG;
  const int64_t E = T * d;
  if (n_src > 1 && src_stride < E) return ATTNRES_ERR_INVALID_ARG;
  const int es = elem_size(v_dtype);
  const Range rv = range_of(V, ((n_src - 1) * (n_src > 1 ? src_stride : 0) + E) * es);
  const Range ro = range_of(out, E * elem_size(out_dtype));
  if (overlap(rv, ro)) return ATTNRES_ERR_INVALID_ARG;
  *a = FullArgs{V, src_stride, n_src, T, d, v_dtype == ATTNRES_BF16, w, gamma, eps, out,
                out_dtype == ATTNRES_BF16, 0};
  a->withhold = withhold_for(kWithholdFull);
  return ATTNRES_OK;
}

int run_full(const FullArgs& a, cudaStream_t s) {
  if (full_fast_ok(a)) return launched([&] { return launch_full_fast(a, s); });
  // General kernel: writes in the storage dtype of the sources.
  if (a.out_bf16 != a.v_bf16) return ATTNRES_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(a.n_src) * 4 > kGenericScoreLimit) return ATTNRES_ERR_UNSUPPORTED;
  MultiArgs m{};
  m.V = a.V;
  m.src_stride = a.src_stride;
  m.n_src = a.n_src;
  m.T = a.T;
  m.d = a.d;
  m.bf16 = a.v_bf16;
  m.W = a.w;
  m.Gamma = a.gamma;
  m.S = 1;
  m.eps = a.eps;
  m.out[0] = a.out;
  m.lse = nullptr;
  m.pre = a.pre;
  m.Q = a.Q;
  return launched([&] { return launch_multi_generic(m, s); });
}

int make_stage1(const void* Src, int64_t src_stride, int32_t n_src, int64_t T, int32_t d,
                int32_t dtype, const float* W, const float* Gamma, int32_t S, float eps,
                void* const* O, float* lse, MultiArgs* m) {
  if (n_src < 1 || d < 1 || T < 0 || !valid_dtype(dtype) || !valid_eps(eps) || S < 1 ||
      S > ATTNRES_MAX_QUERIES)
    return ATTNRES_ERR_INVALID_ARG;
  if (T == 0) return ATTNRES_OK;
  if (!Src || !W || !Gamma || !O) return ATTNRES_ERR_INVALID_ARG;
  const int64_t E = T * d;
  if (n_src > 1 && src_stride < E) return ATTNRES_ERR_INVALID_ARG;
  const int es = elem_size(dtype);
  const Range rs = range_of(Src, ((n_src - 1) * (n_src > 1 ? src_stride : 0) + E) * es);
  const Range rl = lse ? range_of(lse, static_cast<int64_t>(S) * T * 4) : Range{};
  if (overlap(rs, rl)) return ATTNRES_ERR_INVALID_ARG;
  for (int j = 0; j < S; ++j) {
    if (!O[j]) return ATTNRES_ERR_INVALID_ARG;
    const Range rj = range_of(O[j], E * es);
    if (overlap(rj, rs) || overlap(rj, rl)) return ATTNRES_ERR_INVALID_ARG;
    for (int q = 0; q < j; ++q)
      if (overlap(rj, range_of(O[q], E * es))) return ATTNRES_ERR_INVALID_ARG;
  }
  *m = MultiArgs{};
  m->V = Src;
  m->src_stride = src_stride;
  m->n_src = n_src;
  m->T = T;
  m->d = d;
  m->bf16 = dtype == ATTNRES_BF16;
  m->W = W;
  m->Gamma = Gamma;
  m->S = S;
  m->eps = eps;
  for (int j = 0; j < S; ++j) m->out[j] = O[j];
  m->lse = lse;
  m->withhold = withhold_for(kWithholdStage1Tc);
  return ATTNRES_OK;
}

int run_stage1(const MultiArgs& m, cudaStream_t s) {
  if (stage1_fast_ok(m)) return launched([&] { return launch_stage1_fast(m, s); });
  if (static_cast<int64_t>(m.n_src) * m.S * 4 > kGenericScoreLimit) return ATTNRES_ERR_UNSUPPORTED;
  return launched([&] { return launch_multi_generic(m, s); });
}

// Checks and fills a merge whose running sum is P_base + the n_parts
// sublayer outputs at F_parts (part_stride apart), stored to P_out if given.
int make_merge_parts(const void* O_j, const float* lse_j, const float* P_base, const void* F_parts,
                     int64_t part_stride, int32_t n_parts, float* P_out, const float* w, const float* gamma,
                     float eps, int64_t T, int32_t d, int32_t dtype, void* out, void* summary_out, MergeArgs* a) {
  // With a summary the parts hold one output more than the running sum.
  const int32_t nf = n_parts + (summary_out ? 1 : 0);
  if (d < 1 || T < 0 || !valid_dtype(dtype) || !valid_eps(eps) || n_parts < 0 || nf > kMaxMergeParts)
    return ATTNRES_ERR_INVALID_ARG;
  if (n_parts == 0 && !P_base) return ATTNRES_ERR_INVALID_ARG;
  if (T == 0) return ATTNRES_OK;
  if (!O_j || !lse_j || !w || !gamma || !out || (nf > 0 && !F_parts)) return ATTNRES_ERR_INVALID_ARG;
  const int64_t E = T * d;
  if (nf > 1 && part_stride < E) return ATTNRES_ERR_INVALID_ARG;
  const int es = elem_size(dtype);
  const Range ro = range_of(O_j, E * es), rl = range_of(lse_j, T * 4), rout = range_of(out, E * es);
  const Range rb = P_base ? range_of(P_base, E * 4) : Range{};
  const Range rf = nf > 0 ? range_of(F_parts, ((nf - 1) * (nf > 1 ? part_stride : 0) + E) * es) : Range{};
  const Range rp = P_out ? range_of(P_out, E * 4) : Range{};
  const Range rs = summary_out ? range_of(summary_out, E * es) : Range{};
  // out, P_out and summary_out are written: they overlap nothing else, except
  // that P_out may be P_base itself (the running sum advanced in place).
  if (overlap(rout, ro) || overlap(rout, rl) || overlap(rout, rb) || overlap(rout, rf) || overlap(rout, rp) ||
      overlap(rout, rs))
    return ATTNRES_ERR_INVALID_ARG;
  if (overlap(rp, ro) || overlap(rp, rl) || overlap(rp, rf) || (overlap(rp, rb) && P_out != P_base) ||
      overlap(rp, rs))
    return ATTNRES_ERR_INVALID_ARG;
  if (overlap(rs, ro) || overlap(rs, rl) || overlap(rs, rb) || overlap(rs, rf)) return ATTNRES_ERR_INVALID_ARG;
  *a = MergeArgs{O_j, lse_j, P_base, F_parts, nf > 1 ? part_stride : 0, n_parts, P_out, w, gamma, eps, T, d,
                 dtype == ATTNRES_BF16, out};
  a->withhold = withhold_for(kWithholdMerge);
  a->summary = summary_out;
  return ATTNRES_OK;
}

// The single-step merge: P (in/out) advanced by f_prev, or started from it.
int make_merge(const void* O_j, const float* lse_j, float* P, const void* f_prev, int32_t p_is_empty,
               const float* w, const float* gamma, float eps, int64_t T, int32_t d, int32_t dtype,
               void* out, MergeArgs* a) {
  if (d < 1 || T < 0 || !valid_dtype(dtype) || !valid_eps(eps)) return ATTNRES_ERR_INVALID_ARG;
  if (!f_prev && p_is_empty) return ATTNRES_ERR_INVALID_ARG;
  if (T == 0) return ATTNRES_OK;
  if (!O_j || !lse_j || !P || !w || !gamma || !out) return ATTNRES_ERR_INVALID_ARG;
  const int64_t E = T * d;
  const int es = elem_size(dtype);
  const Range ro = range_of(O_j, E * es), rl = range_of(lse_j, T * 4), rp = range_of(P, E * 4),
              rf = f_prev ? range_of(f_prev, E * es) : Range{}, rout = range_of(out, E * es);
  if (overlap(rout, ro) || overlap(rout, rp) || overlap(rout, rf) || overlap(rout, rl) ||
      overlap(rp, ro) || overlap(rp, rf) || overlap(rp, rl))
    return ATTNRES_ERR_INVALID_ARG;
  return make_merge_parts(O_j, lse_j, p_is_empty ? nullptr : P, f_prev, 0, f_prev ? 1 : 0, f_prev ? P : nullptr, w,
                          gamma, eps, T, d, dtype, out, nullptr, a);
}

// Checks and fills a running-sum step: P_base + the n_parts outputs, into
// P_out (fp32) or, rounded, into summary.
int make_accum_parts(const float* P_base, const void* F_parts, int64_t part_stride, int32_t n_parts, float* P_out,
                     void* summary, int64_t T, int32_t d, int32_t dtype, AccumArgs* a) {
  if (d < 1 || T < 0 || !valid_dtype(dtype) || n_parts < 1 || n_parts > kMaxMergeParts)
    return ATTNRES_ERR_INVALID_ARG;
  if (T == 0) return ATTNRES_OK;
  if (!F_parts || (!summary && !P_out)) return ATTNRES_ERR_INVALID_ARG;
  const int64_t E = T * d;
  if (n_parts > 1 && part_stride < E) return ATTNRES_ERR_INVALID_ARG;
  const int es = elem_size(dtype);
  const Range rb = P_base ? range_of(P_base, E * 4) : Range{};
  const Range rf = range_of(F_parts, ((n_parts - 1) * (n_parts > 1 ? part_stride : 0) + E) * es);
  const Range rs = summary ? range_of(summary, E * es) : Range{};
  const Range rp = !summary ? range_of(P_out, E * 4) : Range{};
  if (overlap(rs, rb) || overlap(rs, rf) || overlap(rp, rf) || (overlap(rp, rb) && P_out != P_base))
    return ATTNRES_ERR_INVALID_ARG;
  *a = AccumArgs{P_base, F_parts, n_parts > 1 ? part_stride : 0, n_parts, summary ? nullptr : P_out, summary, T, d,
                 dtype == ATTNRES_BF16};
  return ATTNRES_OK;
}

int make_accum(float* P, const void* f, int32_t p_is_empty, void* summary_out, int64_t T, int32_t d,
               int32_t dtype, AccumArgs* a) {
  if (d < 1 || T < 0 || !valid_dtype(dtype)) return ATTNRES_ERR_INVALID_ARG;
  if (T == 0) return ATTNRES_OK;
  const bool p_used = !(p_is_empty && summary_out);
  if (!f || (p_used && !P)) return ATTNRES_ERR_INVALID_ARG;
  const int64_t E = T * d;
  const int es = elem_size(dtype);
  const Range rp = P ? range_of(P, E * 4) : Range{}, rf = range_of(f, E * es),
              rs = summary_out ? range_of(summary_out, E * es) : Range{};
  if (overlap(rp, rf) || overlap(rs, rf) || overlap(rs, rp)) return ATTNRES_ERR_INVALID_ARG;
  return make_accum_parts(p_is_empty ? nullptr : P, f, 0, 1, P, summary_out, T, d, dtype, a);
}

// Which running sums a Block pass stores (see attnres_block_running_sum_plan):
// stored[j] for 1 <= j < S. Position j (1 <= j <= S) needs P_j, the sum of
// the block's first j outputs; position S is the freeze. Bytes per element
// beyond the fixed O_j / out / summary traffic: each output re-read costs es,
// a stored sum costs 4 to write and 4 to read back. Minimised over all
// choices (dynamic programming over the last stored position); among equal
// costs the plan with fewer stored sums wins, then the one found first.
void running_sum_plan(int S, int es, int* stored) {
  for (int j = 0; j <= S; ++j) stored[j] = 0;
  constexpr int kMax = ATTNRES_MAX_QUERIES + 1;
  int64_t best[kMax];
  int nst[kMax], prev[kMax];
  // Cost of positions m'+1 .. j with base m' and nothing stored between.
  auto run_cost = [&](int mp, int j) {
    int64_t c = 0;
    for (int q = mp + 1; q <= j; ++q) c += static_cast<int64_t>(es) * (q - mp) + (mp > 0 ? 4 : 0);
    return c;
  };
  best[0] = 0;
  nst[0] = 0;
  prev[0] = -1;
  for (int m = 1; m < S; ++m) {
    best[m] = -1;
    for (int mp = 0; mp < m; ++mp) {
      const int64_t c = best[mp] + run_cost(mp, m) + 4;
      if (best[m] < 0 || c < best[m] || (c == best[m] && nst[mp] + 1 < nst[m])) {
        best[m] = c;
        nst[m] = nst[mp] + 1;
        prev[m] = mp;
      }
    }
  }
  int64_t cost = -1;
  int last = 0, n_last = 0;
  for (int mp = 0; mp < S; ++mp) {
    const int64_t c = best[mp] + run_cost(mp, S);
    if (cost < 0 || c < cost || (c == cost && nst[mp] < n_last)) {
      cost = c;
      last = mp;
      n_last = nst[mp];
    }
  }
  for (int m = last; m > 0; m = prev[m]) stored[m] = 1;
}

}  // namespace

extern "C" {

int attnres_abi_version(void) { return 1; }

const char* attnres_status_string(int32_t status) {
  switch (status) {
    case ATTNRES_OK: return "ok";
    case ATTNRES_ERR_INVALID_ARG: return "invalid argument";
    case ATTNRES_ERR_UNSUPPORTED: return "unsupported: beyond a stated limit";
    case ATTNRES_ERR_CUDA: return "CUDA error while launching";
    case ATTNRES_ERR_TIMEOUT: return "a device-side wait ran out of time";
    default: return "unknown status";
  }
}

int attnres_full_fwd(const void* V, int64_t src_stride, int32_t n_src, int64_t T, int32_t d,
                     int32_t v_dtype, const float* w, const float* gamma, float eps, void* out,
                     int32_t out_dtype, void* stream) {
  FullArgs a{};
  const int st = make_full(V, src_stride, n_src, T, d, v_dtype, w, gamma, eps, out, out_dtype, &a);
  if (st != ATTNRES_OK || T == 0) return st;
  return run_full(a, as_stream(stream));
}

int attnres_full_pass(const void* V, int64_t src_stride, int32_t R, int64_t T, int32_t d,
                      int32_t v_dtype, const float* W, const float* Gamma, float eps, void* out,
                      int64_t out_stride, int32_t out_dtype, void* stream) {
  if (R < 1 || d < 1 || T < 0 || !valid_dtype(v_dtype) || !valid_dtype(out_dtype) || !valid_eps(eps))
    return ATTNRES_ERR_INVALID_ARG;
  if (T == 0) return ATTNRES_OK;
  if (!V || !W || !Gamma || !out) return ATTNRES_ERR_INVALID_ARG;
  const int64_t E = T * d;
  if (src_stride < E || out_stride < E) return ATTNRES_ERR_INVALID_ARG;
  const Range rv = range_of(V, ((R - 1) * src_stride + E) * elem_size(v_dtype));
  const Range ro = range_of(out, ((R - 1) * out_stride + E) * elem_size(out_dtype));
  if (overlap(rv, ro)) return ATTNRES_ERR_INVALID_ARG;
  const int oes = elem_size(out_dtype);
  // When no read writes what a later read reads (sources, W and Gamma apart
  // from the outputs), reads after the first overlap the one before them.
  const Range rw = range_of(W, static_cast<int64_t>(R) * d * 4);
  const Range rg = range_of(Gamma, static_cast<int64_t>(R) * d * 4);
  const bool independent = !overlap(rw, ro) && !overlap(rg, ro);
  for (int32_t r = 0; r < R; ++r) {
    FullArgs a{};
    int st = make_full(V, src_stride, r + 1, T, d, v_dtype, W + static_cast<int64_t>(r) * d,
                       Gamma + static_cast<int64_t>(r) * d, eps, static_cast<char*>(out) + r * out_stride * oes,
                       out_dtype, &a);
    if (st != ATTNRES_OK) return st;
    a.late_wait = independent && r > 0;
    st = run_full(a, as_stream(stream));
    if (st != ATTNRES_OK) return st;
  }
  return ATTNRES_OK;
}

// Adds the sublayer pre-norm to a Full read's arguments: out_normed gets
// gamma_pre * z / rms(z); out (z itself) may then be null. Checked like out.
int add_prenorm(const void* V, int64_t src_stride, int32_t n_src, int64_t T, int32_t d, int32_t v_dtype,
                const float* gamma_pre, float eps_pre, void* out, void* out_normed, int32_t out_dtype,
                FullArgs* a) {
  if (!gamma_pre || !out_normed || !valid_eps(eps_pre)) return ATTNRES_ERR_INVALID_ARG;
  const int64_t E = T * d;
  const Range rv = range_of(V, ((n_src - 1) * (n_src > 1 ? src_stride : 0) + E) * elem_size(v_dtype));
  const Range rn = range_of(out_normed, E * elem_size(out_dtype));
  const Range ro = out ? range_of(out, E * elem_size(out_dtype)) : Range{};
  if (overlap(rn, rv) || overlap(rn, ro)) return ATTNRES_ERR_INVALID_ARG;
  a->pre = PreNorm{gamma_pre, eps_pre, out_normed};
  a->out = out;
  return ATTNRES_OK;
}

int attnres_full_fwd_prenorm(const void* V, int64_t src_stride, int32_t n_src, int64_t T, int32_t d,
                             int32_t v_dtype, const float* w, const float* gamma, float eps,
                             const float* gamma_pre, float eps_pre, void* out, void* out_normed,
                             int32_t out_dtype, void* stream) {
  FullArgs a{};
  // make_full checks the read against whichever output is given.
  int st = make_full(V, src_stride, n_src, T, d, v_dtype, w, gamma, eps, out ? out : out_normed, out_dtype, &a);
  if (st != ATTNRES_OK || T == 0) return st;
  st = add_prenorm(V, src_stride, n_src, T, d, v_dtype, gamma_pre, eps_pre, out, out_normed, out_dtype, &a);
  if (st != ATTNRES_OK) return st;
  return run_full(a, as_stream(stream));
}

int attnres_full_pass_prenorm(const void* V, int64_t src_stride, int32_t R, int64_t T, int32_t d,
                              int32_t v_dtype, const float* W, const float* Gamma, float eps,
                              const float* Gamma_pre, float eps_pre, void* out, void* out_normed,
                              int64_t out_stride, int32_t out_dtype, void* stream) {
  if (R < 1 || d < 1 || T < 0 || !valid_dtype(v_dtype) || !valid_dtype(out_dtype) || !valid_eps(eps) ||
      !valid_eps(eps_pre))
    return ATTNRES_ERR_INVALID_ARG;
  if (T == 0) return ATTNRES_OK;
  if (!V || !W || !Gamma || !Gamma_pre || !out_normed) return ATTNRES_ERR_INVALID_ARG;
  const int64_t E = T * d;
  if (src_stride < E || out_stride < E) return ATTNRES_ERR_INVALID_ARG;
  const int oes = elem_size(out_dtype);
  const Range rv = range_of(V, ((R - 1) * src_stride + E) * elem_size(v_dtype));
  const Range rn = range_of(out_normed, ((R - 1) * out_stride + E) * oes);
  const Range ro = out ? range_of(out, ((R - 1) * out_stride + E) * oes) : Range{};
  if (overlap(rv, rn) || overlap(rv, ro) || overlap(rn, ro)) return ATTNRES_ERR_INVALID_ARG;
  const Range rw = range_of(W, static_cast<int64_t>(R) * d * 4);
  const Range rg = range_of(Gamma, static_cast<int64_t>(R) * d * 4);
  const Range rq = range_of(Gamma_pre, static_cast<int64_t>(R) * d * 4);
  const bool independent = !overlap(rw, ro) && !overlap(rg, ro) && !overlap(rq, ro) && !overlap(rw, rn) &&
                           !overlap(rg, rn) && !overlap(rq, rn);
  for (int32_t r = 0; r < R; ++r) {
    void* o = out ? static_cast<char*>(out) + r * out_stride * oes : nullptr;
    void* on = static_cast<char*>(out_normed) + r * out_stride * oes;
    FullArgs a{};
    int st = make_full(V, src_stride, r + 1, T, d, v_dtype, W + static_cast<int64_t>(r) * d,
                       Gamma + static_cast<int64_t>(r) * d, eps, o ? o : on, out_dtype, &a);
    if (st != ATTNRES_OK) return st;
    st = add_prenorm(V, src_stride, r + 1, T, d, v_dtype, Gamma_pre + static_cast<int64_t>(r) * d, eps_pre, o, on,
                     out_dtype, &a);
    if (st != ATTNRES_OK) return st;
    a.late_wait = independent && r > 0;
    st = run_full(a, as_stream(stream));
    if (st != ATTNRES_OK) return st;
  }
  return ATTNRES_OK;
}

int attnres_query_projection(const void* H, int64_t T, int32_t d, int32_t h_dtype, const void* Wq, float* Q,
                             void* stream) {
  if (d < 1 || T < 0 || !valid_dtype(h_dtype)) return ATTNRES_ERR_INVALID_ARG;
  if (h_dtype != ATTNRES_BF16) return ATTNRES_ERR_UNSUPPORTED;
  if (T == 0) return ATTNRES_OK;
  if (!H || !Wq || !Q) return ATTNRES_ERR_INVALID_ARG;
  const Range rq = range_of(Q, T * d * 4);
  if (overlap(rq, range_of(H, T * d * 2)) || overlap(rq, range_of(Wq, static_cast<int64_t>(d) * d * 2)))
    return ATTNRES_ERR_INVALID_ARG;
  cudaStream_t s = as_stream(stream);
  if (proj_tc_ok(H, Wq, Q, T, d)) return launched([&] { return launch_proj_tensor(H, Wq, Q, T, d, s); });
  return launched([&] {
    return proj_ok(H, Wq, Q, d) ? launch_proj(H, Wq, Q, T, d, s) : launch_proj_generic(H, Wq, Q, T, d, s);
  });
}

int attnres_full_fwd_dynq(const void* V, int64_t src_stride, int32_t n_src, int64_t T, int32_t d, int32_t v_dtype,
                          const float* Q, const float* gamma, float eps, void* out, int32_t out_dtype,
                          void* stream) {
  FullArgs a{};
  // make_full checks the read; the shared query argument is unused here.
  int st = make_full(V, src_stride, n_src, T, d, v_dtype, gamma, gamma, eps, out, out_dtype, &a);
  if (st != ATTNRES_OK || T == 0) return st;
  if (!Q) return ATTNRES_ERR_INVALID_ARG;
  if (overlap(range_of(Q, T * d * 4), range_of(out, T * d * elem_size(out_dtype)))) return ATTNRES_ERR_INVALID_ARG;
  a.w = nullptr;
  a.Q = Q;
  return run_full(a, as_stream(stream));
}

int attnres_rmsnorm(const void* x, int64_t T, int32_t d, int32_t dtype, const float* gamma, float eps, void* out,
                    void* stream) {
  if (d < 1 || T < 0 || !valid_dtype(dtype) || !valid_eps(eps)) return ATTNRES_ERR_INVALID_ARG;
  if (T == 0) return ATTNRES_OK;
  if (!x || !gamma || !out) return ATTNRES_ERR_INVALID_ARG;
  const int64_t bytes = T * d * elem_size(dtype);
  // In place (out == x) is allowed; a partial overlap is not.
  if (out != x && overlap(range_of(x, bytes), range_of(out, bytes))) return ATTNRES_ERR_INVALID_ARG;
  return launched([&] { return launch_rmsnorm(x, T, d, dtype == ATTNRES_BF16, gamma, eps, out, as_stream(stream)); });
}

int attnres_full_bwd(const void* V, int64_t src_stride, int32_t n_src, int64_t T, int32_t d,
                     int32_t v_dtype, const float* w, const float* gamma, float eps, const void* dz,
                     int32_t dz_dtype, float* dV, int64_t dv_stride, float* dw, float* dgamma,
                     void* stream) {
  if (n_src < 1 || d < 1 || T < 0 || !valid_dtype(v_dtype) || !valid_dtype(dz_dtype) || !valid_eps(eps))
    return ATTNRES_ERR_INVALID_ARG;
  if (T == 0) return ATTNRES_OK;
  if (!V || !w || !gamma || !dz || !dV) return ATTNRES_ERR_INVALID_ARG;
  const int64_t E = T * d;
  if (n_src > 1 && (src_stride < E || dv_stride < E)) return ATTNRES_ERR_INVALID_ARG;
  const int64_t sstr = n_src > 1 ? src_stride : 0, dstr = n_src > 1 ? dv_stride : 0;
  const Range rv = range_of(V, ((n_src - 1) * sstr + E) * elem_size(v_dtype));
  const Range rz = range_of(dz, E * elem_size(dz_dtype));
  const Range rd = range_of(dV, ((n_src - 1) * dstr + E) * 4);
  const Range rw = dw ? range_of(dw, static_cast<int64_t>(d) * 4) : Range{};
  const Range rg = dgamma ? range_of(dgamma, static_cast<int64_t>(d) * 4) : Range{};
  const Range rq = range_of(w, static_cast<int64_t>(d) * 4), rk = range_of(gamma, static_cast<int64_t>(d) * 4);
  if (overlap(rd, rv) || overlap(rd, rz) || overlap(rd, rw) || overlap(rd, rg) || overlap(rd, rq) ||
      overlap(rd, rk) || overlap(rw, rg) || overlap(rw, rv) || overlap(rg, rv) || overlap(rw, rz) ||
      overlap(rg, rz) || overlap(rw, rq) || overlap(rw, rk) || overlap(rg, rq) || overlap(rg, rk))
    return ATTNRES_ERR_INVALID_ARG;
  const BwdArgs a{V, sstr, n_src, T, d, v_dtype == ATTNRES_BF16, w, gamma, eps, dz, dz_dtype == ATTNRES_BF16,
                  dV, dstr, dw, dgamma};
  const bool fast = full_bwd_fast_ok(a);
  if (!fast && d > kMaxBwdGenericD) return ATTNRES_ERR_UNSUPPORTED;
  return launched([&] { return launch_full_bwd(a, as_stream(stream), fast); });
}

int64_t attnres_block_bwd_scratch_floats(int32_t N, int32_t S, int64_t T, int32_t d) {
  if (N < 1 || S < 1 || T < 0 || d < 1) return -1;
  return (2 * static_cast<int64_t>(N + 1) + S + 1) * T * d;
}

int attnres_block_bwd(const void* Src, int64_t src_stride, const void* F, int64_t f_stride, int32_t N, int32_t S,
                      int64_t T, int32_t d, int32_t dtype, const float* W, const float* Gamma, float eps,
                      const void* dOut, int64_t dout_stride, int32_t dout_dtype, float* dEmb, float* dF,
                      int64_t df_stride, float* dW, float* dGamma, float* scratch, int64_t scratch_floats,
                      void* stream) {
  if (N < 1 || S < 1 || d < 1 || T < 0 || !valid_dtype(dtype) || !valid_dtype(dout_dtype) || !valid_eps(eps))
    return ATTNRES_ERR_INVALID_ARG;
  if (T == 0) return ATTNRES_OK;
  if (!Src || !F || !W || !Gamma || !dOut || !dEmb || !dF || !scratch) return ATTNRES_ERR_INVALID_ARG;
  const int64_t E = T * d;
  const int64_t L = static_cast<int64_t>(N) * S;
  if ((N > 1 && src_stride < E) || (L > 1 && (f_stride < E || dout_stride < E || df_stride < E)))
    return ATTNRES_ERR_INVALID_ARG;
  if (scratch_floats < attnres_block_bwd_scratch_floats(N, S, T, d)) return ATTNRES_ERR_INVALID_ARG;
  const int es = elem_size(dtype);
  const Range rS = range_of(Src, ((N - 1) * (N > 1 ? src_stride : 0) + E) * es);
  const Range rF = range_of(F, ((L - 1) * (L > 1 ? f_stride : 0) + E) * es);
  const Range rZ = range_of(dOut, ((L - 1) * (L > 1 ? dout_stride : 0) + E) * elem_size(dout_dtype));
  const Range rE = range_of(dEmb, E * 4);
  const Range rD = range_of(dF, ((L - 1) * (L > 1 ? df_stride : 0) + E) * 4);
  const Range rW = dW ? range_of(dW, L * d * 4) : Range{};
  const Range rG = dGamma ? range_of(dGamma, L * d * 4) : Range{};
  const Range rX = range_of(scratch, attnres_block_bwd_scratch_floats(N, S, T, d) * 4);
  const Range rq = range_of(W, L * d * 4), rk = range_of(Gamma, L * d * 4);
  const Range outs[] = {rE, rD, rW, rG, rX};
  const Range ins[] = {rS, rF, rZ, rq, rk};
  for (int i = 0; i < 5; ++i) {
    for (int j = 0; j < 5; ++j)
      if (overlap(outs[i], ins[j])) return ATTNRES_ERR_INVALID_ARG;
    for (int j = i + 1; j < 5; ++j)
      if (overlap(outs[i], outs[j])) return ATTNRES_ERR_INVALID_ARG;
  }
  cudaStream_t s = as_stream(stream);
  {
    // Batched: each block's S reads in one pass over the tokens; the sources'
    // gradients (embedding and summaries) gather in the scratch's first N rows.
    BlockBwdArgs b{Src, N > 1 ? src_stride : 0, F, L > 1 ? f_stride : 0, W, Gamma, dOut,
                   L > 1 ? dout_stride : 0, dout_dtype == ATTNRES_BF16, scratch, E, dF, L > 1 ? df_stride : 0,
                   dW, dGamma, N, S, 0, T, d, dtype == ATTNRES_BF16, eps};
    if (block_bwd_batched_ok(b)) {
      if (launched([&] { return cudaMemsetAsync(scratch, 0, N * E * 4, s); }) != ATTNRES_OK) return ATTNRES_ERR_CUDA;
      for (int32_t n = N - 1; n >= 0; --n) {
        b.n = n;
        const int st = launched([&] { return launch_block_bwd_batched(b, s); });
        if (st != ATTNRES_OK) return st;
      }
      return launched([&] { return launch_spread(dEmb, 0, 1, scratch, E, s); });
    }
  }
  // Scratch: fp32 sources Vs [N + 1][E] (embedding, b_1 .. b_{N-1}, and the
  // slot after block n's sources that holds its running sum), their
  // gradients dVs [N + 1][E], the running sums Ps [S][E] (Ps[j] = P of the
  // block's sublayer j), and G [E], the running sum's gradient over the later
  // reads of the block.
  float* Vs = scratch;
  float* dVs = Vs + (N + 1) * E;
  float* Ps = dVs + (N + 1) * E;
  float* G = Ps + static_cast<int64_t>(S) * E;
  const char* Fb = static_cast<const char*>(F);
  const char* Zb = static_cast<const char*>(dOut);
  const int is_bf16 = dtype == ATTNRES_BF16;
  if (launched([&] { return cudaMemsetAsync(dVs, 0, (N + 1) * E * 4, s); }) != ATTNRES_OK) return ATTNRES_ERR_CUDA;
  int st = launched([&] { return launch_widen_rows(Src, N > 1 ? src_stride : 0, is_bf16, Vs, N, E, s); });
  if (st != ATTNRES_OK) return st;
  for (int32_t n = N - 1; n >= 0; --n) {
    const int64_t k0 = static_cast<int64_t>(n) * S;
    // The gradient of b_{n+1}, complete now that every later block is done,
    // goes to each member of block n; its slot then holds block n's running sum.
    if (n + 1 < N) {
      st = launched([&] { return launch_spread(dF + k0 * df_stride, df_stride, S, dVs + (n + 1) * E, E, s); });
      if (st != ATTNRES_OK) return st;
      if (launched([&] { return cudaMemsetAsync(dVs + (n + 1) * E, 0, E * 4, s); }) != ATTNRES_OK)
        return ATTNRES_ERR_CUDA;
    }
    // Running sums as the forward formed them: P_1 = f_{k0}, P_j = P_{j-1} + f_{k0+j-1}.
    for (int32_t j = 1; j < S; ++j) {
      st = launched([&] {
        return launch_psum(Ps + j * E, j == 1 ? nullptr : Ps + (j - 1) * E, Fb + (k0 + j - 1) * f_stride * es,
                           is_bf16, E, s);
      });
      if (st != ATTNRES_OK) return st;
    }
    if (launched([&] { return cudaMemsetAsync(G, 0, E * 4, s); }) != ATTNRES_OK) return ATTNRES_ERR_CUDA;
    for (int32_t j = S - 1; j >= 0; --j) {
      const int64_t k = k0 + j;
      if (j >= 1 && launched([&] {
                      return cudaMemcpyAsync(Vs + (n + 1) * E, Ps + j * E, E * 4, cudaMemcpyDeviceToDevice, s);
                    }) != ATTNRES_OK)
        return ATTNRES_ERR_CUDA;
      st = attnres_full_bwd(Vs, E, n + 1 + (j >= 1 ? 1 : 0), T, d, ATTNRES_F32, W + k * d, Gamma + k * d, eps,
                            Zb + k * dout_stride * elem_size(dout_dtype), dout_dtype, dVs, E,
                            dW ? dW + k * d : nullptr, dGamma ? dGamma + k * d : nullptr, stream);
      if (st != ATTNRES_OK) return st;
      if (j >= 1) {
        st = launched([&] { return launch_gupdate(G, dVs + (n + 1) * E, dF + (k - 1) * df_stride, E, s); });
        if (st != ATTNRES_OK) return st;
      }
    }
  }
  return launched([&] { return launch_spread(dEmb, 0, 1, dVs, E, s); });
}

// Shared checks of the two d-split calls: the shard's sources and queries.
int make_dsplit(const void* Src, int64_t src_stride, int32_t n_src, int64_t T, int32_t d_shard, int32_t d_total,
                int32_t dtype, const float* W, const float* Gamma, int32_t S, float eps, float* partials,
                DsplitArgs* a) {
  if (n_src < 1 || d_shard < 1 || d_total < d_shard || T < 0 || !valid_dtype(dtype) || !valid_eps(eps) || S < 1 ||
      S > ATTNRES_MAX_QUERIES)
    return ATTNRES_ERR_INVALID_ARG;
  if (T == 0) return ATTNRES_OK;
  if (!Src || !partials) return ATTNRES_ERR_INVALID_ARG;
  const int64_t E = T * d_shard;
  if (n_src > 1 && src_stride < E) return ATTNRES_ERR_INVALID_ARG;
  const Range rs = range_of(Src, ((n_src - 1) * (n_src > 1 ? src_stride : 0) + E) * elem_size(dtype));
  const Range rp = range_of(partials, static_cast<int64_t>(n_src) * (S + 1) * T * 4);
  if (overlap(rs, rp)) return ATTNRES_ERR_INVALID_ARG;
  *a = DsplitArgs{};
  a->Src = Src;
  a->src_stride = n_src > 1 ? src_stride : 0;
  a->n_src = n_src;
  a->T = T;
  a->d_shard = d_shard;
  a->d_total = d_total;
  a->bf16 = dtype == ATTNRES_BF16;
  a->W = W;
  a->Gamma = Gamma;
  a->S = S;
  a->eps = eps;
  a->partials = partials;
  return ATTNRES_OK;
}

int attnres_stage1_dsplit_partials(const void* Src, int64_t src_stride, int32_t n_src, int64_t T, int32_t d_shard,
                                   int32_t dtype, const float* W, const float* Gamma, int32_t S, float* partials,
                                   int32_t accumulate, void* stream) {
  DsplitArgs a;
  const int st = make_dsplit(Src, src_stride, n_src, T, d_shard, d_shard, dtype, W, Gamma, S, 0.f, partials, &a);
  if (st != ATTNRES_OK || T == 0) return st;
  if (!W || !Gamma) return ATTNRES_ERR_INVALID_ARG;
  a.accumulate = accumulate != 0;
  if (!dsplit_ok(a)) return ATTNRES_ERR_UNSUPPORTED;
  return launched([&] { return launch_dsplit_partials(a, as_stream(stream)); });
}

int attnres_stage1_dsplit_finish(const void* Src, int64_t src_stride, int32_t n_src, int64_t T, int32_t d_shard,
                                 int32_t d_total, int32_t dtype, const float* partials, int32_t S, float eps,
                                 void* const* O, float* lse, void* stream) {
  DsplitArgs a;
  const int st = make_dsplit(Src, src_stride, n_src, T, d_shard, d_total, dtype, nullptr, nullptr, S, eps,
                             const_cast<float*>(partials), &a);
  if (st != ATTNRES_OK || T == 0) return st;
  if (!O) return ATTNRES_ERR_INVALID_ARG;
  const int64_t E = T * d_shard;
  const int es = elem_size(dtype);
  const Range rs = range_of(Src, ((n_src - 1) * a.src_stride + E) * es);
  const Range rp = range_of(partials, static_cast<int64_t>(n_src) * (S + 1) * T * 4);
  const Range rl = lse ? range_of(lse, static_cast<int64_t>(S) * T * 4) : Range{};
  if (overlap(rl, rs) || overlap(rl, rp)) return ATTNRES_ERR_INVALID_ARG;
  for (int j = 0; j < S; ++j) {
    if (!O[j]) return ATTNRES_ERR_INVALID_ARG;
    const Range ro = range_of(O[j], E * es);
    if (overlap(ro, rs) || overlap(ro, rp) || overlap(ro, rl)) return ATTNRES_ERR_INVALID_ARG;
    for (int q = 0; q < j; ++q)
      if (overlap(ro, range_of(O[q], E * es))) return ATTNRES_ERR_INVALID_ARG;
    a.out[j] = O[j];
  }
  a.lse = lse;
  if (!dsplit_ok(a)) return ATTNRES_ERR_UNSUPPORTED;
  return launched([&] { return launch_dsplit_finish(a, as_stream(stream)); });
}

int attnres_block_stage1(const void* Src, int64_t src_stride, int32_t n_src, int64_t T, int32_t d,
                         int32_t dtype, const float* W, const float* Gamma, int32_t S, float eps,
                         void* const* O, float* lse, void* stream) {
  MultiArgs m{};
  const int st = make_stage1(Src, src_stride, n_src, T, d, dtype, W, Gamma, S, eps, O, lse, &m);
  if (st != ATTNRES_OK || T == 0) return st;
  return run_stage1(m, as_stream(stream));
}

int attnres_block_merge(const void* O_j, const float* lse_j, float* P, const void* f_prev,
                        int32_t p_is_empty, const float* w, const float* gamma, float eps, int64_t T,
                        int32_t d, int32_t dtype, void* out, void* stream) {
  MergeArgs a{};
  const int st = make_merge(O_j, lse_j, P, f_prev, p_is_empty, w, gamma, eps, T, d, dtype, out, &a);
  if (st != ATTNRES_OK || T == 0) return st;
  return launched([&] { return launch_merge(a, as_stream(stream), merge_fast_ok(a)); });
}

int attnres_block_merge_prenorm(const void* O_j, const float* lse_j, float* P, const void* f_prev,
                                int32_t p_is_empty, const float* w, const float* gamma, float eps,
                                const float* gamma_pre, float eps_pre, int64_t T, int32_t d, int32_t dtype,
                                void* out, void* out_normed, void* stream) {
  if (!gamma_pre || !out_normed || !valid_eps(eps_pre)) return ATTNRES_ERR_INVALID_ARG;
  MergeArgs a{};
  // make_merge checks the merge against whichever output is given.
  int st = make_merge(O_j, lse_j, P, f_prev, p_is_empty, w, gamma, eps, T, d, dtype, out ? out : out_normed, &a);
  if (st != ATTNRES_OK || T == 0) return st;
  if (out) {
    const int64_t E = T * d;
    const int es = elem_size(dtype);
    const Range rn = range_of(out_normed, E * es);
    if (overlap(rn, range_of(out, E * es)) || overlap(rn, range_of(O_j, E * es)) ||
        overlap(rn, range_of(P, E * 4)) || overlap(rn, range_of(lse_j, T * 4)) ||
        (f_prev && overlap(rn, range_of(f_prev, E * es))))
      return ATTNRES_ERR_INVALID_ARG;
  }
  a.out = out;
  a.pre = PreNorm{gamma_pre, eps_pre, out_normed};
  return launched([&] { return launch_merge(a, as_stream(stream), merge_fast_ok(a)); });
}

int attnres_block_merge_parts(const void* O_j, const float* lse_j, const float* P_base, const void* F_parts,
                              int64_t part_stride, int32_t n_parts, float* P_out, const float* w,
                              const float* gamma, float eps, int64_t T, int32_t d, int32_t dtype, void* out,
                              void* summary_out, void* stream) {
  MergeArgs a{};
  const int st = make_merge_parts(O_j, lse_j, P_base, F_parts, part_stride, n_parts, P_out, w, gamma, eps, T, d,
                                  dtype, out, summary_out, &a);
  if (st != ATTNRES_OK || T == 0) return st;
  return launched([&] { return launch_merge(a, as_stream(stream), merge_fast_ok(a)); });
}

int attnres_block_summary_parts(const float* P_base, const void* F_parts, int64_t part_stride, int32_t n_parts,
                                float* P_out, void* summary_out, int64_t T, int32_t d, int32_t dtype,
                                void* stream) {
  AccumArgs a{};
  const int st = make_accum_parts(P_base, F_parts, part_stride, n_parts, P_out, summary_out, T, d, dtype, &a);
  if (st != ATTNRES_OK || T == 0) return st;
  return launched([&] { return launch_accum(a, as_stream(stream), accum_fast_ok(a)); });
}

int attnres_block_running_sum_plan(int32_t S, int32_t dtype, int32_t* stored) {
  if (S < 1 || S > ATTNRES_MAX_QUERIES || !valid_dtype(dtype) || !stored) return ATTNRES_ERR_INVALID_ARG;
  int plan[ATTNRES_MAX_QUERIES + 1];
  running_sum_plan(S, elem_size(dtype), plan);
  for (int j = 0; j <= S; ++j) stored[j] = plan[j];
  return ATTNRES_OK;
}

int attnres_block_summary_accumulate(float* P, const void* f, int32_t p_is_empty, void* summary_out,
                                     int64_t T, int32_t d, int32_t dtype, void* stream) {
  AccumArgs a{};
  const int st = make_accum(P, f, p_is_empty, summary_out, T, d, dtype, &a);
  if (st != ATTNRES_OK || T == 0) return st;
  return launched([&] { return launch_accum(a, as_stream(stream), accum_fast_ok(a)); });
}

int attnres_block_pass(const void* F, int64_t f_stride, int32_t N, int32_t S, int64_t T, int32_t d,
                       int32_t dtype, const float* W, const float* Gamma, float eps, void* Src,
                       int64_t src_stride, int32_t freeze_last, void* O_scratch, float* lse_scratch,
                       float* P_scratch, void* out, int64_t out_stride, void* stream) {
  if (N < 1 || S < 1 || S > ATTNRES_MAX_QUERIES || d < 1 || T < 0 || !valid_dtype(dtype) ||
      !valid_eps(eps))
    return ATTNRES_ERR_INVALID_ARG;
  if (T == 0) return ATTNRES_OK;
  if (!F || !W || !Gamma || !Src || !lse_scratch || !out || (S > 1 && (!O_scratch || !P_scratch)))
    return ATTNRES_ERR_INVALID_ARG;
  const int64_t E = T * d;
  if (f_stride < E || src_stride < E || out_stride < E) return ATTNRES_ERR_INVALID_ARG;
  const int es = elem_size(dtype);
  const int64_t L = static_cast<int64_t>(N) * S;
  const int nsrc_slots = N + (freeze_last ? 1 : 0);
  const Range rF = range_of(F, ((L - 1) * f_stride + E) * es);
  const Range rS = range_of(Src, ((nsrc_slots - 1) * src_stride + E) * es);
  const Range rO = S > 1 ? range_of(O_scratch, (S - 1) * E * es) : Range{};
  const Range rL = range_of(lse_scratch, S * T * 4);
  const Range rP = S > 1 || P_scratch ? range_of(P_scratch, E * 4) : Range{};
  const Range rOut = range_of(out, ((L - 1) * out_stride + E) * es);
  const Range all[] = {rF, rS, rO, rL, rP, rOut};
  for (int i = 0; i < 6; ++i)
    for (int j = i + 1; j < 6; ++j)
      if (overlap(all[i], all[j])) return ATTNRES_ERR_INVALID_ARG;

  char* outb = static_cast<char*>(out);
  const char* Fb = static_cast<const char*>(F);
  char* Srcb = static_cast<char*>(Src);
  char* Ob = static_cast<char*>(O_scratch);
  // Which running sums P_j are kept in P_scratch; the others are formed from
  // the last kept one (or from nothing) plus the block's outputs since then.
  int plan[ATTNRES_MAX_QUERIES + 1];
  running_sum_plan(S, es, plan);
  for (int32_t n = 0; n < N; ++n) {
    const int64_t k0 = static_cast<int64_t>(n) * S;  // first sublayer of the block
    // Stage 1: the block's S queries over embedding + n completed block sums.
    void* O[ATTNRES_MAX_QUERIES];
    O[0] = outb + k0 * out_stride * es;
    for (int j = 1; j < S; ++j) O[j] = Ob + (j - 1) * E * es;
    int st = attnres_block_stage1(Src, src_stride, n + 1, T, d, dtype, W + k0 * d, Gamma + k0 * d, S, eps,
                                  O, lse_scratch, stream);
    if (st != ATTNRES_OK) return st;
    // Stage 2: merge each later sublayer's read with its running sum P_j =
    // P_m + f_{k0+m} + ... + f_{k0+j-1}, m the last kept position (0: none).
    // Each read sees only what a layer-by-layer forward has at that point:
    // merge j the outputs f_0 .. f_{j-1}, the freeze the block's last output
    // too. (A merge can also freeze the summary when the caller holds the
    // next output already, attnres_block_merge_parts' summary_out; a model
    // makes f_{S-1} from the last merge's result, so the pass does not.)
    int m = 0;
    for (int j = 1; j < S; ++j) {
      MergeArgs a{};
      st = make_merge_parts(O[j], lse_scratch + j * T, m > 0 ? P_scratch : nullptr, Fb + (k0 + m) * f_stride * es,
                            f_stride, j - m, plan[j] ? P_scratch : nullptr, W + (k0 + j) * d, Gamma + (k0 + j) * d,
                            eps, T, d, dtype, outb + (k0 + j) * out_stride * es, nullptr, &a);
      if (st != ATTNRES_OK) return st;
      // The merge before this one writes neither O[j] nor any output f;
      // stage 1 (before merge 1) writes O[j] but no output f.
      a.early = j >= 2 ? 1 : 2;
      st = launched([&] { return launch_merge(a, as_stream(stream), merge_fast_ok(a)); });
      if (st != ATTNRES_OK) return st;
      if (plan[j]) m = j;
    }
    // Freeze the block summary b_{n+1} = P_S into Src[n + 1]. After a merge it
    // reads the outputs and a kept sum from before that merge, and the merge
    // neither writes those nor reads Src[n + 1]; it lets the freeze start only
    // once it has waited for the kernel before it. So the freeze need not
    // wait, unless the last merge kept the sum it reads.
    if (n + 1 < N || freeze_last) {
      AccumArgs a{};
      st = make_accum_parts(m > 0 ? P_scratch : nullptr, Fb + (k0 + m) * f_stride * es, f_stride, S - m, nullptr,
                            Srcb + (n + 1) * src_stride * es, T, d, dtype, &a);
      if (st != ATTNRES_OK) return st;
      a.no_wait = S > 1 && !plan[S - 1];
      st = launched([&] { return launch_accum(a, as_stream(stream), accum_fast_ok(a)); });
      if (st != ATTNRES_OK) return st;
    }
  }
  return ATTNRES_OK;
}

int attnres_device_status(void* stream) {
  cudaError_t e = stream ? cudaStreamSynchronize(as_stream(stream)) : cudaDeviceSynchronize();
  if (e != cudaSuccess) {
    cudaGetLastError();
    return ATTNRES_ERR_CUDA;
  }
  unsigned int f1 = 0, f2 = 0, f3 = 0, f4 = 0, f5 = 0, f6 = 0, f7 = 0, f8 = 0;
  if (take_timeout_full(&f1) != cudaSuccess || take_timeout_stage1(&f2) != cudaSuccess ||
      take_timeout_merge(&f3) != cudaSuccess || take_timeout_stage1tc(&f4) != cudaSuccess ||
      take_timeout_bwd(&f5) != cudaSuccess || take_timeout_proj(&f6) != cudaSuccess ||
      take_timeout_dsplit(&f7) != cudaSuccess || take_timeout_blockbwd(&f8) != cudaSuccess) {
    cudaGetLastError();
    return ATTNRES_ERR_CUDA;
  }
  if (f1 || f2 || f3 || f4 || f5 || f6 || f7 || f8) return ATTNRES_ERR_TIMEOUT;
  e = cudaGetLastError();
  return e == cudaSuccess ? ATTNRES_OK : ATTNRES_ERR_CUDA;
}

int64_t attnres_test_fail_launch(int64_t after) {
  return g_fail_after.exchange(after < 0 ? -1 : after);
}

int attnres_test_withhold_stage(int32_t kernel, int64_t index) {
  if (kernel < kWithholdNone || kernel > kWithholdMerge || (kernel != kWithholdNone && index < 0))
    return ATTNRES_ERR_INVALID_ARG;
  g_withhold_index.store(kernel == kWithholdNone ? -1 : index);
  g_withhold_kernel.store(kernel);
  return ATTNRES_OK;
}

int attnres_selftest_wait_timeout(void* stream) {
  return launched([&] { return launch_wait_timeout_selftest(as_stream(stream)); });
}

int attnres_kernel_path(int32_t op, const void* src, const void* out, int32_t n_or_s, int32_t s,
                        int64_t T, int32_t d, int32_t dtype) {
  if (!valid_dtype(dtype) || d < 1 || T < 0) return -1;
  // Only alignment is inspected, so an aligned non-null stand-in serves for
  // the fp32 parameter pointers; it is never dereferenced.
  const float* wp = reinterpret_cast<const float*>(static_cast<uintptr_t>(256));
  const int64_t E = T * d;
  switch (op) {
    case 0: {
      FullArgs a{src, E, n_or_s, T, d, dtype == ATTNRES_BF16, wp, wp, 0.f, const_cast<void*>(out),
                 dtype == ATTNRES_BF16};
      return full_fast_ok(a) ? 1 : 0;
    }
    case 1: {
      if (s < 1 || s > ATTNRES_MAX_QUERIES) return -1;
      MultiArgs m{};
      m.V = src;
      m.src_stride = E;
      m.n_src = n_or_s;
      m.T = T;
      m.d = d;
      m.bf16 = dtype == ATTNRES_BF16;
      m.W = wp;
      m.Gamma = wp;
      m.S = s;
      for (int j = 0; j < s; ++j) m.out[j] = const_cast<void*>(out);
      return stage1_fast_ok(m) ? 1 : 0;
    }
    case 2: {
      MergeArgs a{src, wp, wp, src, 0, 1, const_cast<float*>(wp), wp, wp, 0.f, T, d, dtype == ATTNRES_BF16,
                  const_cast<void*>(out)};
      return merge_fast_ok(a) ? 1 : 0;
    }
    case 3: {
      AccumArgs a{wp, src, 0, 1, nullptr, const_cast<void*>(out), T, d, dtype == ATTNRES_BF16};
      return accum_fast_ok(a) ? 1 : 0;
    }
    case 4:
      if (dtype != ATTNRES_BF16) return -1;
      return proj_path(src, src, reinterpret_cast<const float*>(out), T, d);
    default: return -1;
  }
}

}  // extern "C"
