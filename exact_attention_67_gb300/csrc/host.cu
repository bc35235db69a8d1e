// host.cu -- attention forward and backward on host-resident tensors
// (attn_fwd_bwd_host, include/exattn.h).  The (batch, head) problems run in
// groups: each group's inputs are copied in on one stream and its results
// copied out on another while other groups' kernels, or later stages of the
// same group, run on one or two compute streams.  Every attention step is
// the library's own entry points on device copies kept in the caller's
// workspace; this file adds only the copies and their ordering.
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <vector>

#include <cuda_runtime.h>

#include "exattn.h"
#include "kernels.cuh"

using exattn::note_cuda;

namespace {

constexpr size_t kAlign = 256;
size_t align_up(size_t x) { return (x + kAlign - 1) & ~(kAlign - 1); }

// Workspace layout: device copies of q, k, v, dO, o, dq, dk, dv (bf16/f16,
// contiguous [B, H, N, d]), lse (fp32 [B, H, N]) and the backward's row terms
// D, one 256-byte-aligned slice per group (any group count up to B*H fits).
struct Layout {
  size_t t[8];  // q, k, v, dO, o, dq, dk, dv
  size_t lse, D, total;
};

Layout layout(int B, int H, int N, int d) {
  Layout L{};
  const size_t elems = static_cast<size_t>(B) * H * N * d, rows = static_cast<size_t>(B) * H * N;
  size_t off = 0;
  for (int i = 0; i < 8; ++i) {
    L.t[i] = off;
    off += align_up(elems * 2);
  }
  L.lse = off;
  off += align_up(rows * 4);
  L.D = off;
  off += align_up(rows * 4 + kAlign * static_cast<size_t>(B) * H);
  L.total = off;
  return L;
}

struct Events {
  std::vector<cudaEvent_t> ev;
  cudaEvent_t make() {
    cudaEvent_t e = nullptr;
    if (note_cuda(cudaEventCreateWithFlags(&e, cudaEventDisableTiming), "cudaEventCreateWithFlags") != cudaSuccess)
      return nullptr;
    ev.push_back(e);
    return e;
  }
  ~Events() {
    for (cudaEvent_t e : ev) cudaEventDestroy(e);  // released once recorded work completes
  }
};

// b waits for the work queued so far on a.
bool order(Events& E, cudaStream_t a, cudaStream_t b) {
  if (a == b) return true;
  cudaEvent_t e = E.make();
  return e && note_cuda(cudaEventRecord(e, a), "cudaEventRecord") == cudaSuccess &&
         note_cuda(cudaStreamWaitEvent(b, e, 0), "cudaStreamWaitEvent") == cudaSuccess;
}

}  // namespace

extern "C" size_t attn_fwd_bwd_host_workspace_size(int B, int H, int N, int d, int causal) {
  if (attn_bwd_workspace_size(B, H, N, d, causal) == 0) return 0;  // invalid sizes
  return layout(B, H, N, d).total;
}

extern "C" int attn_fwd_bwd_host(int dtype, const void* q, const void* k, const void* v, const void* dO, void* o,
                                 float* lse, void* dq, void* dk, void* dv, int B, int H, int N, int d, int causal,
                                 float scale, void* workspace, size_t workspace_bytes, int groups, void* stream,
                                 void* copy_in_stream, void* copy_out_stream, void* stream2) {
  if (!q || !k || !v || !dO || !o || !lse || !dq || !dk || !dv) return EXATTN_ERR_NULL;
  if (dtype != EXATTN_DTYPE_BF16 && dtype != EXATTN_DTYPE_F16) return EXATTN_ERR_UNSUPPORTED;
  const size_t need = attn_fwd_bwd_host_workspace_size(B, H, N, d, causal);
  if (need == 0) return (d != 64 && d != 128) ? EXATTN_ERR_UNSUPPORTED : EXATTN_ERR_SHAPE;
  if (!std::isfinite(scale) || !(scale > 0.f)) return EXATTN_ERR_VALUE;
  if (groups < 1) return EXATTN_ERR_VALUE;
  if (!workspace || workspace_bytes < need) return EXATTN_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(workspace) % 16 != 0) return EXATTN_ERR_ALIGN;

  const int BH = B * H;
  const int G = std::min(groups, BH);
  const Layout L = layout(B, H, N, d);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  const cudaStream_t sin = copy_in_stream ? static_cast<cudaStream_t>(copy_in_stream) : s;
  const cudaStream_t sout = copy_out_stream ? static_cast<cudaStream_t>(copy_out_stream) : s;
  const cudaStream_t s2 = stream2 ? static_cast<cudaStream_t>(stream2) : s;
  const size_t row_bytes = static_cast<size_t>(N) * d * 2;  // one (batch, head) problem of one tensor
  const void* hin[4] = {q, k, v, dO};
  void* hout[4] = {o, dq, dk, dv};
  auto dev_t = [&](int i, int a) { return ws + L.t[i] + static_cast<size_t>(a) * row_bytes; };
  auto dev_lse = [&](int a) { return reinterpret_cast<float*>(ws + L.lse) + static_cast<size_t>(a) * N; };
  auto host_in = [&](int i, int a) { return static_cast<const uint8_t*>(hin[i]) + static_cast<size_t>(a) * row_bytes; };

  Events E;
  // Earlier work on `stream` may still use the workspace or the host buffers.
  if (!order(E, s, sin) || !order(E, s, sout) || !order(E, s, s2)) return EXATTN_ERR_CUDA;
  std::vector<cudaEvent_t> ev_qkv(G), ev_do(G);
  for (int g = 0; g < G; ++g) {  // inputs in use order: Q, K, V of a group (forward), then its dO (backward)
    const int a = static_cast<int>(static_cast<long long>(g) * BH / G);
    const int b = static_cast<int>(static_cast<long long>(g + 1) * BH / G);
    for (int i = 0; i < 4; ++i) {
      if (note_cuda(cudaMemcpyAsync(dev_t(i, a), host_in(i, a), (b - a) * row_bytes, cudaMemcpyHostToDevice, sin),
                    "cudaMemcpyAsync (host to device)") != cudaSuccess)
        return EXATTN_ERR_CUDA;
      if (i == 2 || i == 3) {
        cudaEvent_t e = E.make();
        if (!e || note_cuda(cudaEventRecord(e, sin), "cudaEventRecord") != cudaSuccess) return EXATTN_ERR_CUDA;
        (i == 2 ? ev_qkv : ev_do)[g] = e;
      }
    }
  }
  const bool bf16 = dtype == EXATTN_DTYPE_BF16;
  size_t d_off = L.D;
  for (int g = 0; g < G; ++g) {
    const int a = static_cast<int>(static_cast<long long>(g) * BH / G);
    const int b = static_cast<int>(static_cast<long long>(g + 1) * BH / G);
    const int n = b - a;  // the group as one batch of n heads
    const cudaStream_t c = (g & 1) ? s2 : s;
    float* D = reinterpret_cast<float*>(ws + d_off);
    d_off += align_up(static_cast<size_t>(n) * N * 4);
    auto copy_out = [&](std::initializer_list<int> which) {
      if (!order(E, c, sout)) return false;
      for (int i : which) {
        const bool is_lse = i < 0;
        void* dst = is_lse ? static_cast<void*>(lse + static_cast<size_t>(a) * N)
                           : static_cast<void*>(static_cast<uint8_t*>(hout[i]) + static_cast<size_t>(a) * row_bytes);
        const void* src = is_lse ? static_cast<const void*>(dev_lse(a)) : static_cast<const void*>(dev_t(4 + i, a));
        const size_t bytes = is_lse ? static_cast<size_t>(n) * N * 4 : n * row_bytes;
        if (note_cuda(cudaMemcpyAsync(dst, src, bytes, cudaMemcpyDeviceToHost, sout),
                      "cudaMemcpyAsync (device to host)") != cudaSuccess)
          return false;
      }
      return true;
    };
    if (note_cuda(cudaStreamWaitEvent(c, ev_qkv[g], 0), "cudaStreamWaitEvent") != cudaSuccess) return EXATTN_ERR_CUDA;
    const exattn_strides cs{static_cast<long long>(n) * N * d, static_cast<long long>(N) * d, d};
    int rc = bf16 ? attn_fwd(dev_t(0, a), dev_t(1, a), dev_t(2, a), dev_t(4, a), dev_lse(a), 1, n, N, d, causal, scale,
                             c)
                  : attn_fwd_ex(dtype, dev_t(0, a), cs, dev_t(1, a), cs, dev_t(2, a), cs, dev_t(4, a), cs, dev_lse(a),
                                1, n, N, d, causal, 0, scale, c);
    if (rc != EXATTN_OK) return rc;
    if (!copy_out({0, -1})) return EXATTN_ERR_CUDA;  // O and lse leave while the backward runs
    if (note_cuda(cudaStreamWaitEvent(c, ev_do[g], 0), "cudaStreamWaitEvent") != cudaSuccess) return EXATTN_ERR_CUDA;
    if (bf16) {
      if ((rc = attn_bwd_preprocess(dev_t(4, a), dev_t(3, a), D, 1, n, N, d, c)) != EXATTN_OK) return rc;
      if ((rc = attn_bwd_dkdv(dev_t(0, a), dev_t(1, a), dev_t(2, a), dev_t(3, a), dev_lse(a), D, dev_t(6, a),
                              dev_t(7, a), 1, n, N, d, causal, scale, c)) != EXATTN_OK)
        return rc;
      if (!copy_out({2, 3})) return EXATTN_ERR_CUDA;  // dK, dV leave while dQ is computed
      if ((rc = attn_bwd_dq(dev_t(0, a), dev_t(1, a), dev_t(2, a), dev_t(3, a), dev_lse(a), D, dev_t(5, a), 1, n, N,
                            d, causal, scale, c)) != EXATTN_OK)
        return rc;
      if (!copy_out({1})) return EXATTN_ERR_CUDA;
    } else {
      if ((rc = attn_bwd_ex(dtype, dev_t(0, a), cs, dev_t(1, a), cs, dev_t(2, a), cs, dev_t(4, a), cs, dev_t(3, a), cs,
                            dev_lse(a), dev_t(5, a), cs, dev_t(6, a), cs, dev_t(7, a), cs, 1, n, N, d, causal, 0,
                            scale, D, align_up(static_cast<size_t>(n) * N * 4), c)) != EXATTN_OK)
        return rc;
      if (!copy_out({1, 2, 3})) return EXATTN_ERR_CUDA;
    }
  }
  // The call's work is complete when everything queued on `stream` so far is.
  if (!order(E, s2, s) || !order(E, sout, s)) return EXATTN_ERR_CUDA;
  return EXATTN_OK;
}
