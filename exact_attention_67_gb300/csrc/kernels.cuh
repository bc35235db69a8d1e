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

// Where the rows of batch b live.  Fixed length (cu_seqlens == nullptr):
// rows [0, N) of batch b, statistics (lse, D) at [b*H + h, N].  Packed
// variable length: sequence b is rows [cu_seqlens[b], cu_seqlens[b+1]) of
// one [total, H, d] tensor (batch stride unused), statistics at [h, total].
struct SeqView {
  const int* cu_seqlens;  // device, B + 1 non-decreasing offsets, or nullptr
  int total;              // rows of the packed tensors
};

// Rows of batch b as seen by one CTA: first row in the tensor, length
// (clamped to [0, n_max] and to the packed tensor, so a bad offset table can
// never send an access out of bounds), the batch coordinate of the tensor
// maps and output strides, and the first statistics index of head h.
struct SeqRows {
  int start, n, b_coord;
  long long stat0;
};

__device__ __forceinline__ SeqRows seq_rows(const SeqView& sv, int b, int h, int H, int n_max) {
  SeqRows r;
  if (!sv.cu_seqlens) {
    r.start = 0;
    r.n = n_max;
    r.b_coord = b;
    r.stat0 = (static_cast<long long>(b) * H + h) * n_max;
  } else {
    const int s0 = min(max(sv.cu_seqlens[b], 0), sv.total);
    const int s1 = min(max(sv.cu_seqlens[b + 1], s0), sv.total);
    r.start = s0;
    r.n = min(s1 - s0, n_max);
    r.b_coord = 0;
    r.stat0 = static_cast<long long>(h) * sv.total + s0;
  }
  return r;
}

// Grid order shared by the attention kernels.  The (batch, head) problems run
// in groups of `group`, sized on the host (l2_group) so that the operand the
// CTAs of one problem all re-read -- K and V for the forward and dQ, Q and dO
// for dK/dV -- stays in L2 for the whole group; within a group the tiles go
// heaviest first (tile 0 is the caller's heaviest) and problems fastest.
// With group == BH this is plain (tile, sub, problem) order.
struct GridPos {
  int tile, sub, bh;
};

__host__ __device__ __forceinline__ GridPos grid_pos(int block, int BH, int n_tiles, int n_sub, int group) {
  const long long b = block;
  const long long per_full = static_cast<long long>(group) * n_tiles * n_sub;
  const long long full = BH / group;  // complete groups
  long long g, r;
  int size;
  if (b < full * per_full) {
    g = b / per_full;
    r = b % per_full;
    size = group;
  } else {
    g = full;
    r = b - full * per_full;
    size = BH - static_cast<int>(full) * group;
  }
  const long long per_tile = static_cast<long long>(size) * n_sub;
  GridPos p;
  p.tile = static_cast<int>(r / per_tile);
  p.sub = static_cast<int>(r % per_tile / size);
  p.bh = static_cast<int>(g * group + r % size);
  return p;
}

// Keys per step of the dQ kernel: 64 at d = 128; 96 at d = 64, where a
// query tile's TMEM (dQ 64 + S 96 + dP 96 columns) still fits two tiles in
// 512 columns and each step's fixed hand-off latencies cover more keys.
constexpr int dq_key_step(int d) { return d == 64 ? 96 : 64; }
// Queries per step of the dK/dV kernel, likewise: 64 at d = 128; 96 at d = 64
// (dK, dV 64 columns each, two buffers of S^T and dP^T of 96 columns).
constexpr int dkdv_query_step(int d) { return d == 64 ? 96 : 64; }

// Problems per group for grid_pos: as many as keep their re-read operands
// (bytes_per_problem each) within `budget` bytes of the 129 MB L2 (half of
// it by default), at least one.
constexpr long long kL2GroupBytes = 64ll << 20;
inline int l2_group(long long bytes_per_problem, int BH, long long budget = kL2GroupBytes) {
  long long g = bytes_per_problem > 0 ? budget / bytes_per_problem : BH;
  if (g > BH) g = BH;
  return g < 1 ? 1 : static_cast<int>(g);
}

// Key side of the forward when it differs from the query side: nk keys per
// problem with the queries aligned to the last nq of them (bottom-right:
// query i sits at key position i + nk - nq), and the keys split over
// n_splits CTAs of tiles_per_split 128-key tiles each.  With part_o set,
// every split writes fp32 partial results that launch_fwd_merge combines:
//   part_o    [n_splits, B*H, nq_pad, d]  O of the split (normalised within it)
//   part_lse  [n_splits, B*H, nq_pad]     logsumexp of the split (for lse)
//   part_lseb [n_splits, B*H, nq_pad]     logsumexp of the rounded weights (for O)
constexpr int kMaxSplits = 512;  // key splits launch_fwd_merge combines at most

struct KvSplit {
  int nk;  // 0: as many keys as queries, no offset
  int n_splits, tiles_per_split, nq_pad;
  float* part_o;
  float* part_lse;
  float* part_lseb;
};

struct FwdArgs {
  const CUtensorMap* tm_q;  // 4-D maps (d, N, H, B), box 64 x 128 x 1 x 1, 128-byte swizzle
  const CUtensorMap* tm_k;
  const CUtensorMap* tm_v;
  void* o;                  // [B, H, N, d] view with strides so
  Strides so;
  float* lse;               // fp32 [B*H, N]
  int N, H, BH, d, causal, dtype;
  int window;               // 0, or W >= 1: key j visible to query i iff i - j < W (and j - i < W if not causal)
  SeqView seq;              // N is the longest sequence when seq.cu_seqlens is set
  KvSplit kv;               // decode-shaped problems (kv.nk > 0); zero otherwise
  float* o32;               // optional fp32 copy of O, contiguous [B*H, N, d] (fixed-length calls), or nullptr
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
  // K and V with a box of dq_key_step(d) rows: the dQ kernel's key tiles
  const CUtensorMap* tm_kdq;
  const CUtensorMap* tm_vdq;
  // Q and dO with a box of dkdv_query_step(d) rows: the dK/dV kernel's query tiles
  const CUtensorMap* tm_qkv;
  const CUtensorMap* tm_dokv;
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
  const float* o32;         // optional fp32 O, contiguous [B*H, N, d]: D_i from it instead of o
  bool dq_computes_D;       // the dQ kernel forms D_i (from o or o32, and dO) and writes it to D
  int N, H, BH, d, causal, dtype;
  int window;               // as FwdArgs::window
  SeqView seq;              // as FwdArgs::seq
  float scale, scale_log2;
  unsigned* err;
  int device;
};

// Records, for the calling host thread, a CUDA call that failed (`driver`:
// `code` is a CUresult, else a cudaError_t); exattn_last_cuda_error() reads
// it back.  note_cuda passes a runtime status through, recording it if it
// is an error.
void note_failure(const char* call, int code, bool driver);
inline cudaError_t note_cuda(cudaError_t e, const char* call) {
  if (e != cudaSuccess) note_failure(call, static_cast<int>(e), false);
  return e;
}

cudaError_t ensure_smem_attr(const void* kernel, int bytes, int device);
cudaError_t launch_fwd(const FwdArgs& a, cudaStream_t stream);
// Combines the split partials of a forward with a.kv.part_o set into O and lse.
cudaError_t launch_fwd_merge(const FwdArgs& a, cudaStream_t stream);
// Decode-shaped forward for at most kDecodeMaxQ queries at d = 128
// (decode.cu): a.tm_q with a box of kDecodeQCols rows, a.kv as for the
// forward's key split (nq_pad = kDecodeQCols, n_splits >= 1; partials in
// a.kv.part_o when n_splits > 1).  Measured faster than the forward kernel
// with split keys up to 12 queries at d = 128, slower at 16.
constexpr int kDecodeMaxQ = 12;
constexpr int kDecodeQCols = 16;  // query columns of the kernel (the MMA's N)
cudaError_t launch_decode(const FwdArgs& a, cudaStream_t stream);
cudaError_t launch_bwd_prep(const BwdArgs& a, cudaStream_t stream);
cudaError_t launch_bwd_dkdv(const BwdArgs& a, cudaStream_t stream);
cudaError_t launch_bwd_dq(const BwdArgs& a, cudaStream_t stream);

}  // namespace exattn
