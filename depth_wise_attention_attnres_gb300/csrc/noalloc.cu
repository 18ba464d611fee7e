// attnres_block_pass_noalloc: the Block AttnRes pass with its workspace in a
// fixed array that the library itself holds, for callers that cannot
// allocate device memory (see include/attnres.h).
//
// The workspace of a pass (stage-1 results O, their log-masses lse and the
// fp32 running sum P) lives in g_noalloc_scratch, a file-scope device array.
// In host code that name is only a stand-in for the symbol, not a device
// address, so the address is obtained with cudaGetSymbolAddress while the
// caller's context is current, and cached per CUDA context. The cache is
// keyed by the context's process-unique id (cuCtxGetId), not by the device
// number: after cudaDeviceReset, or once a primary context is released and
// made again, the module loads anew, the array may sit elsewhere, and the
// next call looks its address up again instead of handing the kernels a
// pointer into memory that is no longer mapped. The entry point then calls
// attnres_block_pass with pointers into the array.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <mutex>
#include <utility>
#include <vector>

#include "attnres.h"

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[ATTNRES_NOALLOC_SCRATCH_BYTES];

std::mutex g_mu;
// (context id, device address of g_noalloc_scratch in that context).
std::vector<std::pair<unsigned long long, void*>> g_scratch_ptrs;

// The driver calls that identify the current context, looked up once.
struct CtxFns {
  PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
  PFN_cuCtxGetId_v12000 get_id = nullptr;
};

bool ctx_fns(CtxFns* out) {
  static CtxFns fns;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fns.get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fns.get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(p);
    cudaGetLastError();
  }
  *out = fns;
  return fns.get_current && fns.get_id;
}

// Id of the current context, or false if there is none yet.
bool current_ctx_id(const CtxFns& f, unsigned long long* id) {
  CUcontext ctx = nullptr;
  if (f.get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return false;
  return f.get_id(ctx, id) == CUDA_SUCCESS;
}

// Device address of g_noalloc_scratch in the current context. The first call
// in a context looks it up (cudaGetSymbolAddress, which also loads this
// file's module into the context when module loading is lazy).
int scratch_address(void** out) {
  std::lock_guard<std::mutex> lk(g_mu);
  CtxFns f;
  if (!ctx_fns(&f)) return ATTNRES_ERR_CUDA;
  unsigned long long id = 0;
  if (current_ctx_id(f, &id)) {
    for (const auto& e : g_scratch_ptrs)
      if (e.first == id) {
        *out = e.second;
        return ATTNRES_OK;
      }
  }
  // Unknown (or not yet created) context: the lookup below makes the
  // runtime's context current if it is not yet.
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
  if (e != cudaSuccess || p == nullptr) {
    cudaGetLastError();
    return ATTNRES_ERR_CUDA;
  }
  if (!current_ctx_id(f, &id)) return ATTNRES_ERR_CUDA;
  bool found = false;
  for (auto& s : g_scratch_ptrs)
    if (s.first == id) {
      s.second = p;
      found = true;
    }
  if (!found) g_scratch_ptrs.emplace_back(id, p);
  *out = p;
  return ATTNRES_OK;
}

unsigned long long round256(unsigned long long x) { return (x + 255ull) & ~255ull; }

}  // namespace

extern "C" int attnres_block_pass_noalloc(const void* F, int64_t f_stride, int32_t N, int32_t S,
                                          int64_t T, int32_t d, int32_t dtype, const float* W,
                                          const float* Gamma, float eps, void* Src, int64_t src_stride,
                                          int32_t freeze_last, void* out, int64_t out_stride,
                                          void* stream) {
  // The argument checks of attnres_block_pass that need no workspace come
  // first, so a call that is both malformed and too large reports the
  // malformed argument.
  if (N < 1 || S < 1 || S > ATTNRES_MAX_QUERIES || d < 1 || T < 0 ||
      (dtype != ATTNRES_F32 && dtype != ATTNRES_BF16) || !(eps >= 0.0f && eps < 3.0e38f))
    return ATTNRES_ERR_INVALID_ARG;
  if (T == 0)  // nothing to do; attnres_block_pass checks the rest
    return attnres_block_pass(F, f_stride, N, S, T, d, dtype, W, Gamma, eps, Src, src_stride,
                              freeze_last, nullptr, nullptr, nullptr, out, out_stride, stream);
  if (!F || !W || !Gamma || !Src || !out) return ATTNRES_ERR_INVALID_ARG;
  const unsigned long long limit = ATTNRES_NOALLOC_SCRATCH_BYTES;
  const unsigned long long t = static_cast<unsigned long long>(T);
  const unsigned long long dd = static_cast<unsigned long long>(d);
  // T or d alone beyond the limit never fits; below it T * d cannot overflow.
  if (t > limit || dd > limit) return ATTNRES_ERR_UNSUPPORTED;
  const unsigned long long E = t * dd;
  const int64_t Ei = static_cast<int64_t>(E);
  if (f_stride < Ei || src_stride < Ei || out_stride < Ei) return ATTNRES_ERR_INVALID_ARG;
  // Workspace: O for queries 1..S-1 and P exist only when S > 1; lse always.
  const unsigned long long es = dtype == ATTNRES_BF16 ? 2ull : 4ull;
  const unsigned long long o_bytes = S > 1 ? round256(static_cast<unsigned long long>(S - 1) * E * es) : 0ull;
  const unsigned long long l_bytes = round256(static_cast<unsigned long long>(S) * t * 4ull);
  const unsigned long long p_bytes = S > 1 ? round256(E * 4ull) : 0ull;
  if (o_bytes + l_bytes + p_bytes > limit) return ATTNRES_ERR_UNSUPPORTED;

  void* base = nullptr;
  const int st = scratch_address(&base);
  if (st != ATTNRES_OK) return st;
  unsigned char* b = static_cast<unsigned char*>(base);
  void* O = S > 1 ? b : nullptr;
  float* lse = reinterpret_cast<float*>(b + o_bytes);
  float* P = S > 1 ? reinterpret_cast<float*>(b + o_bytes + l_bytes) : nullptr;
  return attnres_block_pass(F, f_stride, N, S, T, d, dtype, W, Gamma, eps, Src, src_stride,
                            freeze_last, O, lse, P, out, out_stride, stream);
}
