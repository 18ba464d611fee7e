// attnres_block_pass_noalloc: the Block AttnRes pass with its workspace in a
// fixed array that the library itself holds, for callers that cannot
// allocate device memory (see include/attnres.h).
//
// The workspace of a pass (stage-1 results O, their log-masses lse and the
// fp32 running sum P) lives in g_noalloc_scratch, a file-scope device array.
// In host code that name is only a stand-in for the symbol, not a device
// address, so the address is obtained once per device with
// cudaGetSymbolAddress while that device is current and cached here. The
// entry point then calls attnres_block_pass with pointers into the array.
#include <cuda_runtime.h>

#include <mutex>

#include "attnres.h"

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[ATTNRES_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_noalloc_scratch on the current device; looked up on
// the first call for each device.
int scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return ATTNRES_ERR_CUDA;
  }
  if (dev < 0 || dev >= kMaxDevices) return ATTNRES_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return ATTNRES_ERR_CUDA;
    }
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return ATTNRES_OK;
}

unsigned long long round256(unsigned long long x) { return (x + 255ull) & ~255ull; }

}  // namespace

extern "C" int attnres_block_pass_noalloc(const void* F, int64_t f_stride, int32_t N, int32_t S,
                                          int64_t T, int32_t d, int32_t dtype, const float* W,
                                          const float* Gamma, float eps, void* Src, int64_t src_stride,
                                          int32_t freeze_last, void* out, int64_t out_stride,
                                          void* stream) {
  if (N < 1 || S < 1 || S > ATTNRES_MAX_QUERIES || d < 1 || T < 0 ||
      (dtype != ATTNRES_F32 && dtype != ATTNRES_BF16))
    return ATTNRES_ERR_INVALID_ARG;
  if (T == 0)  // nothing to do; attnres_block_pass checks the rest
    return attnres_block_pass(F, f_stride, N, S, T, d, dtype, W, Gamma, eps, Src, src_stride,
                              freeze_last, nullptr, nullptr, nullptr, out, out_stride, stream);
  // Workspace: O for queries 1..S-1 and P exist only when S > 1; lse always.
  const unsigned long long limit = ATTNRES_NOALLOC_SCRATCH_BYTES;
  const unsigned long long es = dtype == ATTNRES_BF16 ? 2ull : 4ull;
  const unsigned long long t = static_cast<unsigned long long>(T);
  const unsigned long long dd = static_cast<unsigned long long>(d);
  if (t > limit || dd > limit || t * dd > limit) return ATTNRES_ERR_UNSUPPORTED;
  const unsigned long long E = t * dd;
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
