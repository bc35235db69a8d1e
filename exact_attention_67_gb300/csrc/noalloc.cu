// noalloc.cu -- attn_bwd_noalloc: the backward pass for callers that cannot
// allocate device memory.
//
// attn_bwd needs a workspace (one fp32 row term D_i per query row) that the
// caller allocates.  Some callers cannot: a plugin handed only the input and
// output buffers by a runtime that owns all device memory, or code on a
// latency-critical path where an allocation (which may synchronise the
// device) is not allowed.  This entry point takes the same inputs and outputs
// but keeps D in a fixed-size array that is part of the loaded library, so it
// calls no cudaMalloc, cudaFree or any other allocating routine.
//
// The array lives in device memory of every GPU that loads the library, for
// as long as the library stays loaded.  Its address is looked up once per
// device (cudaGetSymbolAddress, with that device current) on the first call
// made on that device; make that first call before any stream capture.  All
// calls share the array and it keeps the previous call's contents: nothing in
// it needs to start at zero (the first backward stage writes every D_i the
// later stages read), but calls whose executions overlap on the GPU (e.g. on
// two streams) race on it and must be serialised by the caller.
#include <mutex>

#include "exattn.h"
#include "kernels.cuh"

namespace exattn {
namespace {

// 16 MiB: D_i for up to 4,194,304 query rows (B * H * N).
constexpr size_t kNoallocRows = size_t(1) << 22;
static __device__ __align__(256) float g_noalloc_scratch[kNoallocRows];

constexpr int kMaxDev = 64;
std::mutex g_noalloc_mu;
float* g_noalloc_ptr[kMaxDev] = {};

// Device address of this device's scratch array (set-up on first use).
int noalloc_scratch(float** out) {
  int dev = 0;
  if (note_cuda(cudaGetDevice(&dev), "cudaGetDevice") != cudaSuccess) return EXATTN_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDev) {
    note_failure("cudaGetDevice (device ordinal out of range)", static_cast<int>(cudaErrorInvalidDevice), false);
    return EXATTN_ERR_CUDA;
  }
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    float* p = nullptr;
    if (note_cuda(cudaGetSymbolAddress(reinterpret_cast<void**>(&p), g_noalloc_scratch), "cudaGetSymbolAddress") !=
            cudaSuccess ||
        !p)
      return EXATTN_ERR_CUDA;
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
  return EXATTN_OK;
}

}  // namespace
}  // namespace exattn

extern "C" int attn_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const void* dO,
                                const float* lse, void* dq, void* dk, void* dv, int B, int H, int N, int d,
                                int causal, float scale, void* stream) {
  if (B >= 1 && H >= 1 && N >= 1 &&
      static_cast<unsigned long long>(B) * H * N > static_cast<unsigned long long>(exattn::kNoallocRows))
    return EXATTN_ERR_WORKSPACE;  // more query rows than the built-in scratch holds
  const size_t need = attn_bwd_workspace_size(B, H, N, d, causal);
  if (need == 0) {
    // invalid shape: let attn_bwd report the precise error before any CUDA call
    return attn_bwd(q, k, v, o, dO, lse, dq, dk, dv, B, H, N, d, causal, scale, nullptr, 0, stream);
  }
  if (!q || !k || !v || !o || !dO || !lse || !dq || !dk || !dv) return EXATTN_ERR_NULL;
  float* scratch = nullptr;
  const int rc = exattn::noalloc_scratch(&scratch);
  if (rc != EXATTN_OK) return rc;
  return attn_bwd(q, k, v, o, dO, lse, dq, dk, dv, B, H, N, d, causal, scale, scratch,
                  exattn::kNoallocRows * sizeof(float), stream);
}
