// merge.cu -- combines the fp32 partial results of a decode-shaped forward
// whose keys were split over CTAs (the forward kernel's key split and the
// decode kernel), for sm_103a.
//
// O and lse of query row r from the key splits' partials: with the splits'
// logsumexps L_s and Lb_s, lse = log sum_s exp(L_s) and O = sum_s exp(Lb_s -
// log sum_s' exp(Lb_s')) O_s -- the logsumexp-weighted combination the online
// softmax applies inside one CTA ("Gemini 3 Flash的注意力内核重写：算子融合如何
// 实现亚毫秒级推理", §3 在线softmax算法), across CTAs.  Both kernels write L_s
// and Lb_s from their sum of the f16-rounded weights (the one normalisation
// the single-CTA forward uses), so L_s = Lb_s; the two inputs are kept in the
// workspace layout.
//
// One block per row: the threads share the splits for the two logsumexps,
// then THREADS / d groups of d threads (one column each) share them for O,
// and the groups' sums are added in shared memory.  A thread loads BATCH of
// its splits' O values at once and adds them round four accumulators, and
// its first batch is loaded before the logsumexps are reduced (the values
// do not depend on them).  With few rows (one long sequence) and many splits
// each block's chain of loads is the whole kernel, so those launches take
// 1024 threads and batches of 16; otherwise the blocks hide each other's
// latency (or there is little to load) and take 256 threads and batches of 4.
#include "kernels.cuh"
#include "ptx.cuh"

namespace exattn {

template <typename T, int D, int THREADS, int BATCH>
__global__ void __launch_bounds__(THREADS) attn_merge_kernel(const float* __restrict__ part_o,
                                                             const float* __restrict__ part_lse,
                                                             const float* __restrict__ part_lseb, int n_splits,
                                                             int nq_pad, int N, int H, int BH,
                                                             T* __restrict__ out, Strides so,
                                                             float* __restrict__ lse_out) {
  constexpr int G = THREADS / D;                            // split groups for the O sum
  constexpr int NW = THREADS / 32;
  constexpr int LPT = (kMaxSplits + THREADS - 1) / THREADS;  // logsumexps per thread
  static_assert(NW <= 32 && THREADS % D == 0, "block reductions and column groups");
  __shared__ float w_s[kMaxSplits];
  __shared__ float red[2][NW];
  __shared__ float acc_g[G][D];
  // Launched as a programmatic dependent of the kernel that wrote the
  // partials: wait until that grid has completed and its writes are visible
  // (without such a launch this returns at once).
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int bh = static_cast<int>(blockIdx.x) / N, row = static_cast<int>(blockIdx.x) % N;
  const int hh = bh % H, bb = bh / H;
  auto at = [&](int s) { return (static_cast<long long>(s) * BH + bh) * nq_pad + row; };
  // Max or sum of (a, b) over the block, the same value and order in every
  // warp: lanes, then the warps' results through shared memory.
  auto block_reduce = [&](float a, float b, bool is_max, float& ra, float& rb) {
    auto op = [&](float x, float y) { return is_max ? fmaxf(x, y) : x + y; };
    for (int o = 16; o > 0; o >>= 1) {
      a = op(a, __shfl_xor_sync(0xffffffffu, a, o));
      b = op(b, __shfl_xor_sync(0xffffffffu, b, o));
    }
    if (lane == 0) {
      red[0][warp] = a;
      red[1][warp] = b;
    }
    __syncthreads();
    const float id = is_max ? -INFINITY : 0.f;
    a = lane < NW ? red[0][lane] : id;
    b = lane < NW ? red[1][lane] : id;
    for (int o = 16; o > 0; o >>= 1) {
      a = op(a, __shfl_xor_sync(0xffffffffu, a, o));
      b = op(b, __shfl_xor_sync(0xffffffffu, b, o));
    }
    ra = a;
    rb = b;
    __syncthreads();
  };
  // This thread's first batch of O values (split s = g + u G, column c).
  const int g = tid / D, c = tid % D;
  const long long split_stride = static_cast<long long>(BH) * nq_pad * D;
  const float* po = part_o + at(0) * D + c;
  float x[BATCH];
#pragma unroll
  for (int u = 0; u < BATCH; ++u) {
    const int s = g + u * G;
    x[u] = s < n_splits ? po[s * split_stride] : 0.f;
  }
  // The splits' logsumexps, loaded once and kept for both reductions.
  float L[LPT], Lb[LPT];
  float mx_l = -INFINITY, mxb_l = -INFINITY;
#pragma unroll
  for (int i = 0; i < LPT; ++i) {
    const int s = tid + i * THREADS;
    L[i] = s < n_splits ? part_lse[at(s)] : -INFINITY;
    Lb[i] = s < n_splits ? part_lseb[at(s)] : -INFINITY;
    mx_l = fmaxf(mx_l, L[i]);
    mxb_l = fmaxf(mxb_l, Lb[i]);
  }
  float mx, mxb;
  block_reduce(mx_l, mxb_l, true, mx, mxb);
  float sum_l = 0.f, sumb_l = 0.f;
#pragma unroll
  for (int i = 0; i < LPT; ++i) {
    const int s = tid + i * THREADS;
    if (L[i] != -INFINITY) sum_l += expf(L[i] - mx);
    const float w = Lb[i] != -INFINITY ? expf(Lb[i] - mxb) : 0.f;
    if (s < n_splits) w_s[s] = w;
    sumb_l += w;
  }
  float sum, sumb;
  block_reduce(sum_l, sumb_l, false, sum, sumb);  // its barriers also publish w_s
  float acc4[4] = {0.f, 0.f, 0.f, 0.f};
  for (int s0 = g;;) {
#pragma unroll
    for (int u = 0; u < BATCH; ++u) {
      const int s = s0 + u * G;
      if (s < n_splits) acc4[u & 3] = fmaf(w_s[s], x[u], acc4[u & 3]);
    }
    s0 += BATCH * G;
    if (s0 >= n_splits) break;
#pragma unroll
    for (int u = 0; u < BATCH; ++u) {
      const int s = s0 + u * G;
      x[u] = s < n_splits ? po[s * split_stride] : 0.f;
    }
  }
  acc_g[g][c] = (acc4[0] + acc4[1]) + (acc4[2] + acc4[3]);
  __syncthreads();
  if (tid < D) {
    float v = 0.f;
#pragma unroll
    for (int k = 0; k < G; ++k) v += acc_g[k][tid];
    v *= sumb > 0.f ? 1.f / sumb : 0.f;
    T* orow = out + bb * so.b + hh * so.h + static_cast<long long>(row) * so.n;
    if constexpr (Elem<T>::kFmt == 1) orow[tid] = __float2bfloat16_rn(v);
    else orow[tid] = __float2half_rn(v);
  }
  if (tid == 0) lse_out[static_cast<long long>(bh) * N + row] = mx + logf(sum);
}

template <typename T, int D>
static cudaError_t launch_merge_t(const FwdArgs& a, cudaStream_t stream) {
  if (a.kv.n_splits < 1 || a.kv.n_splits > kMaxSplits)
    return note_cuda(cudaErrorInvalidValue, "split merge (key split count)");
  const long long rows = static_cast<long long>(a.BH) * a.N;
  int sms = 0;
  const cudaError_t e =
      note_cuda(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, a.device), "cudaDeviceGetAttribute");
  if (e != cudaSuccess) return e;
  // A programmatic dependent launch: the blocks can be resident (waiting in
  // griddepcontrol.wait) when the partials' last writer finishes, which
  // hides this launch's latency behind it.
  const bool wide = rows < 2ll * sms && a.kv.n_splits > 16;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(rows));
  cfg.blockDim = dim3(wide ? 1024 : 256);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t le =
      wide ? cudaLaunchKernelEx(&cfg, attn_merge_kernel<T, D, 1024, 16>, a.kv.part_o, a.kv.part_lse, a.kv.part_lseb,
                                a.kv.n_splits, a.kv.nq_pad, a.N, a.H, a.BH, static_cast<T*>(a.o), a.so, a.lse)
           : cudaLaunchKernelEx(&cfg, attn_merge_kernel<T, D, 256, 4>, a.kv.part_o, a.kv.part_lse, a.kv.part_lseb,
                                a.kv.n_splits, a.kv.nq_pad, a.N, a.H, a.BH, static_cast<T*>(a.o), a.so, a.lse);
  const cudaError_t last = cudaGetLastError();  // also clears a launch error le reported
  return note_cuda(le != cudaSuccess ? le : last, "split-merge kernel launch");
}

cudaError_t launch_fwd_merge(const FwdArgs& a, cudaStream_t stream) {
  if (a.dtype == kF16) return a.d == 64 ? launch_merge_t<__half, 64>(a, stream) : launch_merge_t<__half, 128>(a, stream);
  return a.d == 64 ? launch_merge_t<__nv_bfloat16, 64>(a, stream) : launch_merge_t<__nv_bfloat16, 128>(a, stream);
}

}  // namespace exattn
