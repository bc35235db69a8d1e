// kernels.cuh -- launch interfaces between the C ABI (api.cu) and the kernels.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>

namespace exattn {

struct FwdArgs {
  const CUtensorMap* tm_q;  // 3-D maps over [B*H, N, d] bf16, box 64 x 128 x 1, 128-byte swizzle
  const CUtensorMap* tm_k;
  const CUtensorMap* tm_v;
  void* o;                  // bf16 [B*H, N, d]
  float* lse;               // fp32 [B*H, N]
  int N, BH, d, causal;
  float scale_log2;         // scale * log2(e)
  unsigned* err;            // device watchdog word
  int device;
};

struct BwdArgs {
  // 3-D maps over [B*H, N, d] bf16 with 128-byte swizzle; box 64 x 128 x 1 ...
  const CUtensorMap* tm_q128;
  const CUtensorMap* tm_k128;
  const CUtensorMap* tm_v128;
  const CUtensorMap* tm_do128;
  // ... and box 64 x 64 x 1
  const CUtensorMap* tm_q64;
  const CUtensorMap* tm_k64;
  const CUtensorMap* tm_v64;
  const CUtensorMap* tm_do64;
  const void* q;            // raw pointers, bf16 [B*H, N, d]
  const void* k;
  const void* v;
  const void* o;
  const void* dO;
  const float* lse;         // fp32 [B*H, N], natural log
  void* dq;
  void* dk;
  void* dv;
  float* D;                 // workspace: fp32 [B*H, N]
  int N, BH, d, causal;
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
