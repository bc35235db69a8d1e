// kernels.cuh -- launch interfaces between the C ABI (api.cu) and the kernels.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>

namespace exattn {

// Element strides of a [B, H, N, d] view whose d axis is contiguous.
struct Strides {
  long long b, h, n;
};

// Element type of Q, K, V, O, dO, dQ, dK, dV (the C ABI's exattn_dtype).
enum : int { kBF16 = 0, kF16 = 1 };

struct FwdArgs {
  const CUtensorMap* tm_q;  // 4-D maps (d, N, H, B), box 64 x 128 x 1 x 1, 128-byte swizzle
  const CUtensorMap* tm_k;
  const CUtensorMap* tm_v;
  void* o;                  // [B, H, N, d] view with strides so
  Strides so;
  float* lse;               // fp32 [B*H, N]
  int N, H, BH, d, causal, dtype;
  int window;               // 0, or W >= 1: key j visible to query i iff i - j < W (and j - i < W if not causal)
  float scale_log2;         // scale * log2(e)
  unsigned* err;            // device watchdog word
  int device;
};

struct BwdArgs {
  // 4-D maps (d, N, H, B) with 128-byte swizzle; box 64 x 128 x 1 x 1 ...
  const CUtensorMap* tm_q128;
  const CUtensorMap* tm_k128;
  const CUtensorMap* tm_v128;
  const CUtensorMap* tm_do128;
  // ... and box 64 x 64 x 1 x 1
  const CUtensorMap* tm_q64;
  const CUtensorMap* tm_k64;
  const CUtensorMap* tm_v64;
  const CUtensorMap* tm_do64;
  const void* o;            // [B, H, N, d] views (d contiguous) with their element strides
  Strides so;
  const void* dO;
  Strides sdo;
  void* dq;
  Strides sdq;
  void* dk;
  Strides sdk;
  void* dv;
  Strides sdv;
  const float* lse;         // fp32 [B*H, N], natural log
  float* D;                 // workspace: fp32 [B*H, N]
  int N, H, BH, d, causal, dtype;
  int window;               // as FwdArgs::window
  float scale, scale_log2;
  unsigned* err;
  int device;
};

cudaError_t ensure_smem_attr(const void* kernel, int bytes, int device);
cudaError_t launch_fwd(const FwdArgs& a, cudaStream_t stream);
cudaError_t launch_bwd_prep(const BwdArgs& a, cudaStream_t stream);
cudaError_t launch_bwd_dkdv(const BwdArgs& a, cudaStream_t stream);
cudaError_t launch_bwd_dq(const BwdArgs& a, cudaStream_t stream);

}  // namespace exattn
