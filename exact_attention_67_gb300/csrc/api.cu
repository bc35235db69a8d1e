// api.cu -- the C ABI of libexattn.so (declared in include/exattn.h):
// argument validation, per-device set-up, TMA tensor-map encoding and kernel
// launches.  No device memory is allocated here and nothing synchronises
// except exattn_device_error().
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "exattn.h"
#include "kernels.cuh"
#include "ptx.cuh"

namespace exattn {

// Watchdog word shared by every kernel launch on a device (bit flags from ptx.cuh).
__device__ unsigned g_err_word;

// One warp waits on an mbarrier that nothing ever arrives on, with the given
// limit: the bounded wait gives up, reports through the watchdog word and the
// kernel returns normally.  Used to check the failure path end to end.
__global__ void watchdog_selftest_kernel(unsigned long long limit_ns, unsigned* err) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncwarp();
  const WaitCtl wc{&abort_flag, err};
  if (threadIdx.x == 0) mbar_wait(&bar, 0, wc, limit_ns);
  __syncwarp();
}

namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
using CtxGetCurrentFn = CUresult (*)(CUcontext*);

constexpr int kMaxDevices = 64;

struct DeviceState {
  bool ready = false;
  int status = EXATTN_OK;  // EXATTN_OK, EXATTN_ERR_ARCH or EXATTN_ERR_CUDA once set up
  unsigned* err = nullptr;
};

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];
EncodeTiledFn g_encode = nullptr;
CtxGetCurrentFn g_ctx_current = nullptr;

struct AttrKey {
  const void* fn;
  int device;
};
AttrKey g_attr_done[256];
int g_attr_count = 0;

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// The last CUDA call that failed on this host thread (exattn_last_cuda_error).
thread_local const char* t_fail_call = nullptr;
thread_local int t_fail_code = 0;
thread_local bool t_fail_driver = false;
thread_local char t_fail_text[192];

// A driver entry point by name (CUDA 12.0 ABI); false if it is missing.
bool driver_fn(const char* name, void** fn) {
  cudaDriverEntryPointQueryResult q;
  if (note_cuda(cudaGetDriverEntryPointByVersion(name, fn, 12000, cudaEnableDefault, &q),
                "cudaGetDriverEntryPointByVersion") != cudaSuccess)
    return false;
  if (q != cudaDriverEntryPointSuccess || !*fn) {
    note_failure("cudaGetDriverEntryPointByVersion (driver entry point not found)", static_cast<int>(q), false);
    return false;
  }
  return true;
}

// Arch check, watchdog address and the driver entry points, once per device;
// then, on every call, the device's primary context made current if the
// calling host thread has none.  A thread that has made no CUDA call yet has
// no current context, and the tensor-map encoder, a driver call, fails in it
// with CUDA_ERROR_INVALID_CONTEXT; cudaSetDevice makes the primary context
// current (the one the kernels already run in).
int device_setup(int* dev_out, unsigned** err_out) {
  int dev = 0;
  if (note_cuda(cudaGetDevice(&dev), "cudaGetDevice") != cudaSuccess) return EXATTN_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) {
    note_failure("cudaGetDevice (device ordinal out of range)", static_cast<int>(cudaErrorInvalidDevice), false);
    return EXATTN_ERR_CUDA;
  }
  int status;
  unsigned* err;
  {
    // Set-up under the lock; afterwards the state is only read.
    std::lock_guard<std::mutex> lk(g_mu);
    DeviceState& st = g_dev[dev];
    if (!st.ready) {
      int major = 0, minor = 0;
      const char* what = "cudaDeviceGetAttribute";
      if (note_cuda(cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev), what) != cudaSuccess ||
          note_cuda(cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev), what) != cudaSuccess)
        return EXATTN_ERR_CUDA;
      if (major != 10 || minor != 3) {
        st.status = EXATTN_ERR_ARCH;
      } else {
        void* p = nullptr;
        if (note_cuda(cudaGetSymbolAddress(&p, g_err_word), "cudaGetSymbolAddress") != cudaSuccess)
          return EXATTN_ERR_CUDA;
        st.err = static_cast<unsigned*>(p);
        if (!g_encode || !g_ctx_current) {
          void *enc = nullptr, *cur = nullptr;
          if (!driver_fn("cuTensorMapEncodeTiled", &enc) || !driver_fn("cuCtxGetCurrent", &cur))
            return EXATTN_ERR_CUDA;
          g_encode = reinterpret_cast<EncodeTiledFn>(enc);
          g_ctx_current = reinterpret_cast<CtxGetCurrentFn>(cur);
        }
        st.status = EXATTN_OK;
      }
      st.ready = true;
    }
    status = st.status;
    err = st.err;
  }
  if (status != EXATTN_OK) return status;
  CUcontext ctx = nullptr;
  const CUresult r = g_ctx_current(&ctx);
  if (r != CUDA_SUCCESS) {
    note_failure("cuCtxGetCurrent", static_cast<int>(r), true);
    return EXATTN_ERR_CUDA;
  }
  if (!ctx && note_cuda(cudaSetDevice(dev), "cudaSetDevice") != cudaSuccess) return EXATTN_ERR_CUDA;
  *dev_out = dev;
  *err_out = err;
  return EXATTN_OK;
}

// A [B, H, N, d] view (d contiguous, element strides s) as a 4-D map
// (d, N, H, B); box = 64 columns (128 bytes) x box_rows rows x 1 x 1.
bool make_map(CUtensorMap* m, const void* base, int dtype, int B, int H, int N, int d, const Strides& s,
              int box_rows) {
  const cuuint64_t dims[4] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(H),
                              static_cast<cuuint64_t>(B)};
  // A stride along an extent-1 axis is never used; give the encoder a legal one.
  const long long sn = N > 1 ? s.n : d, sh = H > 1 ? s.h : d, sb = B > 1 ? s.b : d;
  const cuuint64_t strides[3] = {static_cast<cuuint64_t>(sn) * 2, static_cast<cuuint64_t>(sh) * 2,
                                 static_cast<cuuint64_t>(sb) * 2};
  const cuuint32_t box[4] = {64, static_cast<cuuint32_t>(box_rows), 1, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  const CUtensorMapDataType ty = dtype == kF16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const CUresult r = g_encode(m, ty, 4, const_cast<void*>(base), dims, strides, box, estr,
                              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) note_failure("cuTensorMapEncodeTiled", static_cast<int>(r), true);
  return r == CUDA_SUCCESS;
}

int check_common(int B, int H, int N, int d, float scale) {
  if (B < 1 || H < 1 || N < 1) return EXATTN_ERR_SHAPE;
  if (static_cast<long long>(B) * H * N >= (1ll << 31)) return EXATTN_ERR_SHAPE;
  if (static_cast<long long>(B) * H >= (1ll << 24)) return EXATTN_ERR_SHAPE;
  if (d != 64 && d != 128) return EXATTN_ERR_UNSUPPORTED;
  if (!std::isfinite(scale) || !(scale > 0.f)) return EXATTN_ERR_VALUE;
  return EXATTN_OK;
}

Strides contiguous(int H, int N, int d) {
  return Strides{static_cast<long long>(H) * N * d, static_cast<long long>(N) * d, static_cast<long long>(d)};
}

Strides to_strides(const exattn_strides& s) { return Strides{s.b_stride, s.h_stride, s.n_stride}; }

// Strides in elements: non-negative, multiples of 8 (16 bytes, the TMA rule),
// below 2^36; positive along every axis of extent > 1.
int check_strides(const exattn_strides& s, int B, int H, int N) {
  const long long v[3] = {s.b_stride, s.h_stride, s.n_stride};
  const int ext[3] = {B, H, N};
  for (int i = 0; i < 3; ++i) {
    if (v[i] < 0 || v[i] >= (1ll << 36) || (v[i] & 7) != 0) return EXATTN_ERR_ALIGN;
    if (ext[i] > 1 && v[i] == 0) return EXATTN_ERR_SHAPE;
  }
  return EXATTN_OK;
}

}  // namespace

void note_failure(const char* call, int code, bool driver) {
  t_fail_call = call;
  t_fail_code = code;
  t_fail_driver = driver;
}

cudaError_t ensure_smem_attr(const void* kernel, int bytes, int device) {
  std::lock_guard<std::mutex> lk(g_mu);
  for (int i = 0; i < g_attr_count; ++i)
    if (g_attr_done[i].fn == kernel && g_attr_done[i].device == device) return cudaSuccess;
  cudaError_t e = note_cuda(cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes),
                            "cudaFuncSetAttribute");
  if (e != cudaSuccess) return e;
  if (g_attr_count < 256) g_attr_done[g_attr_count++] = AttrKey{kernel, device};
  return cudaSuccess;
}

}  // namespace exattn

using namespace exattn;

namespace {

// Tensor maps cover [map_b, H, map_n, d]: the batch itself, or (packed
// variable-length sequences, seq.cu_seqlens set) one batch of seq.total rows.
int fwd_impl(int dtype, const void* q, const Strides& sq, const void* k, const Strides& sk, const void* v,
             const Strides& sv, void* o, const Strides& so, float* lse, int B, int H, int N, int d, int causal,
             int window, float scale, void* stream, const SeqView& seq = SeqView{nullptr, 0},
             float* o32 = nullptr) {
  int dev = 0;
  unsigned* err = nullptr;
  int rc = device_setup(&dev, &err);
  if (rc != EXATTN_OK) return rc;
  const int map_b = seq.cu_seqlens ? 1 : B, map_n = seq.cu_seqlens ? seq.total : N;
  CUtensorMap mq, mk, mv;
  if (!make_map(&mq, q, dtype, map_b, H, map_n, d, sq, 128) || !make_map(&mk, k, dtype, map_b, H, map_n, d, sk, 128) ||
      !make_map(&mv, v, dtype, map_b, H, map_n, d, sv, 128))
    return EXATTN_ERR_CUDA;
  FwdArgs a{};
  a.tm_q = &mq;
  a.tm_k = &mk;
  a.tm_v = &mv;
  a.o = o;
  a.so = so;
  a.lse = lse;
  a.N = N;
  a.H = H;
  a.BH = B * H;
  a.d = d;
  a.causal = causal ? 1 : 0;
  a.dtype = dtype;
  a.window = window;
  a.seq = seq;
  a.o32 = o32;
  a.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  a.err = err;
  a.device = dev;
  return launch_fwd(a, static_cast<cudaStream_t>(stream)) == cudaSuccess ? EXATTN_OK : EXATTN_ERR_CUDA;
}

}  // namespace

extern "C" int attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int d,
                        int causal, float scale, void* stream) {
  if (!q || !k || !v || !o || !lse) return EXATTN_ERR_NULL;
  int rc = check_common(B, H, N, d, scale);
  if (rc != EXATTN_OK) return rc;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) || !aligned(lse, 4))
    return EXATTN_ERR_ALIGN;
  const Strides c = contiguous(H, N, d);
  return fwd_impl(kBF16, q, c, k, c, v, c, o, c, lse, B, H, N, d, causal, 0, scale, stream);
}

extern "C" int attn_fwd_ex(int dtype, const void* q, exattn_strides sq, const void* k, exattn_strides sk,
                           const void* v, exattn_strides sv, void* o, exattn_strides so, float* lse, int B, int H,
                           int N, int d, int causal, int window, float scale, void* stream) {
  if (!q || !k || !v || !o || !lse) return EXATTN_ERR_NULL;
  if (dtype != EXATTN_DTYPE_BF16 && dtype != EXATTN_DTYPE_F16) return EXATTN_ERR_UNSUPPORTED;
  int rc = check_common(B, H, N, d, scale);
  if (rc != EXATTN_OK) return rc;
  if (window < 0) return EXATTN_ERR_VALUE;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) || !aligned(lse, 4))
    return EXATTN_ERR_ALIGN;
  const exattn_strides* all[4] = {&sq, &sk, &sv, &so};
  for (const exattn_strides* s : all)
    if ((rc = check_strides(*s, B, H, N)) != EXATTN_OK) return rc;
  return fwd_impl(dtype == EXATTN_DTYPE_F16 ? kF16 : kBF16, q, to_strides(sq), k, to_strides(sk), v, to_strides(sv),
                  o, to_strides(so), lse, B, H, N, d, causal, window, scale, stream);
}

extern "C" int attn_fwd_o32(int dtype, const void* q, exattn_strides sq, const void* k, exattn_strides sk,
                            const void* v, exattn_strides sv, void* o, exattn_strides so, float* lse, float* o32,
                            int B, int H, int N, int d, int causal, int window, float scale, void* stream) {
  if (!o32) return EXATTN_ERR_NULL;
  if (!aligned(o32, 16)) return EXATTN_ERR_ALIGN;
  if (!q || !k || !v || !o || !lse) return EXATTN_ERR_NULL;
  if (dtype != EXATTN_DTYPE_BF16 && dtype != EXATTN_DTYPE_F16) return EXATTN_ERR_UNSUPPORTED;
  int rc = check_common(B, H, N, d, scale);
  if (rc != EXATTN_OK) return rc;
  if (window < 0) return EXATTN_ERR_VALUE;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) || !aligned(lse, 4))
    return EXATTN_ERR_ALIGN;
  const exattn_strides* all[4] = {&sq, &sk, &sv, &so};
  for (const exattn_strides* s : all)
    if ((rc = check_strides(*s, B, H, N)) != EXATTN_OK) return rc;
  return fwd_impl(dtype == EXATTN_DTYPE_F16 ? kF16 : kBF16, q, to_strides(sq), k, to_strides(sk), v, to_strides(sv),
                  o, to_strides(so), lse, B, H, N, d, causal, window, scale, stream, SeqView{nullptr, 0}, o32);
}

extern "C" size_t attn_bwd_workspace_size(int B, int H, int N, int d, int causal) {
  (void)causal;
  if (check_common(B, H, N, d, 1.f) != EXATTN_OK) return 0;
  const size_t rows = static_cast<size_t>(B) * H * N;
  return (rows * sizeof(float) + 255) & ~size_t(255);
}

namespace {

// Shared set-up of the backward entry points (arguments already validated):
// device state, the tensor maps of the given inputs (a null input skips its
// maps), and the launch arguments.
struct BwdMaps {
  // 128-row boxes of q, k, v, dO; 64-row boxes; k, v in the dQ kernel's key
  // steps and q, dO in the dK/dV kernel's query steps where those are 96.
  CUtensorMap m[12];
};

struct BwdInputs {
  const void* p[4];  // q, k, v, dO (any may be null)
  Strides s[4];
};

int bwd_setup(BwdArgs& a, BwdMaps& maps, int dtype, const BwdInputs& in, int B, int H, int N, int d, int causal,
              float scale, int window = 0, const SeqView& seq = SeqView{nullptr, 0}) {
  int dev = 0;
  unsigned* err = nullptr;
  int rc = device_setup(&dev, &err);
  if (rc != EXATTN_OK) return rc;
  const int map_b = seq.cu_seqlens ? 1 : B, map_n = seq.cu_seqlens ? seq.total : N;
  for (int i = 0; i < 4; ++i) {
    if (!in.p[i]) continue;
    if (!make_map(&maps.m[i], in.p[i], dtype, map_b, H, map_n, d, in.s[i], 128) ||
        !make_map(&maps.m[4 + i], in.p[i], dtype, map_b, H, map_n, d, in.s[i], 64))
      return EXATTN_ERR_CUDA;
  }
  const int kstep = dq_key_step(d);
  const bool own_kv_maps = kstep != 64 && kstep != 128;
  for (int i = 1; own_kv_maps && i < 3; ++i) {
    if (in.p[i] && !make_map(&maps.m[7 + i], in.p[i], dtype, map_b, H, map_n, d, in.s[i], kstep))
      return EXATTN_ERR_CUDA;
  }
  a.tm_kdq = own_kv_maps ? &maps.m[8] : (kstep == 64 ? &maps.m[5] : &maps.m[1]);
  a.tm_vdq = own_kv_maps ? &maps.m[9] : (kstep == 64 ? &maps.m[6] : &maps.m[2]);
  const int qstep = dkdv_query_step(d);
  const bool own_q_maps = qstep != 64 && qstep != 128;
  for (int i = 0; own_q_maps && i < 4; i += 3) {  // q and dO
    if (in.p[i] && !make_map(&maps.m[i == 0 ? 10 : 11], in.p[i], dtype, map_b, H, map_n, d, in.s[i], qstep))
      return EXATTN_ERR_CUDA;
  }
  a.tm_qkv = own_q_maps ? &maps.m[10] : (qstep == 64 ? &maps.m[4] : &maps.m[0]);
  a.tm_dokv = own_q_maps ? &maps.m[11] : (qstep == 64 ? &maps.m[7] : &maps.m[3]);
  a.tm_q128 = &maps.m[0];
  a.tm_k128 = &maps.m[1];
  a.tm_v128 = &maps.m[2];
  a.tm_do128 = &maps.m[3];
  a.tm_q64 = &maps.m[4];
  a.tm_k64 = &maps.m[5];
  a.tm_v64 = &maps.m[6];
  a.tm_do64 = &maps.m[7];
  a.N = N;
  a.H = H;
  a.BH = B * H;
  a.d = d;
  a.causal = causal ? 1 : 0;
  a.dtype = dtype;
  a.window = window;
  a.seq = seq;
  a.scale = scale;
  a.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  a.err = err;
  a.device = dev;
  return EXATTN_OK;
}

BwdInputs contiguous_inputs(const void* q, const void* k, const void* v, const void* dO, int H, int N, int d) {
  const Strides c = contiguous(H, N, d);
  return BwdInputs{{q, k, v, dO}, {c, c, c, c}};
}

// The whole backward on one stream: the dQ kernel, which also forms the row
// terms D_i and stores them in the workspace, then dK/dV, which reads them.
int bwd_impl(int dtype, const BwdInputs& in, const void* o, const Strides& so, const Strides& sdo, const float* lse,
             void* dq, const Strides& sdq, void* dk, const Strides& sdk, void* dv, const Strides& sdv, int B, int H,
             int N, int d, int causal, int window, float scale, void* workspace, void* stream,
             const SeqView& seq = SeqView{nullptr, 0}, const float* o32 = nullptr) {
  BwdArgs a{};
  BwdMaps maps;
  int rc = bwd_setup(a, maps, dtype, in, B, H, N, d, causal, scale, window, seq);
  if (rc != EXATTN_OK) return rc;
  a.o = o;
  a.so = so;
  a.dO = in.p[3];
  a.sdo = sdo;
  a.lse = lse;
  a.dq = dq;
  a.sdq = sdq;
  a.dk = dk;
  a.sdk = sdk;
  a.dv = dv;
  a.sdv = sdv;
  a.D = static_cast<float*>(workspace);
  a.o32 = o32;
  a.dq_computes_D = true;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (launch_bwd_dq(a, st) != cudaSuccess) return EXATTN_ERR_CUDA;
  if (launch_bwd_dkdv(a, st) != cudaSuccess) return EXATTN_ERR_CUDA;
  return EXATTN_OK;
}

}  // namespace

extern "C" int attn_bwd_preprocess(const void* o, const void* dO, float* D, int B, int H, int N, int d,
                                   void* stream) {
  if (!o || !dO || !D) return EXATTN_ERR_NULL;
  int rc = check_common(B, H, N, d, 1.f);
  if (rc != EXATTN_OK) return rc;
  if (!aligned(o, 16) || !aligned(dO, 16) || !aligned(D, 4)) return EXATTN_ERR_ALIGN;
  BwdArgs a{};
  BwdMaps maps;
  const BwdInputs none = contiguous_inputs(nullptr, nullptr, nullptr, nullptr, H, N, d);
  if ((rc = bwd_setup(a, maps, kBF16, none, B, H, N, d, 0, 1.f)) != EXATTN_OK) return rc;
  a.o = o;
  a.so = contiguous(H, N, d);
  a.dO = dO;
  a.sdo = a.so;
  a.D = D;
  return launch_bwd_prep(a, static_cast<cudaStream_t>(stream)) == cudaSuccess ? EXATTN_OK : EXATTN_ERR_CUDA;
}

extern "C" int attn_bwd_dkdv(const void* q, const void* k, const void* v, const void* dO, const float* lse,
                             const float* D, void* dk, void* dv, int B, int H, int N, int d, int causal, float scale,
                             void* stream) {
  if (!q || !k || !v || !dO || !lse || !D || !dk || !dv) return EXATTN_ERR_NULL;
  int rc = check_common(B, H, N, d, scale);
  if (rc != EXATTN_OK) return rc;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(dO, 16) || !aligned(dk, 16) ||
      !aligned(dv, 16) || !aligned(lse, 4) || !aligned(D, 4))
    return EXATTN_ERR_ALIGN;
  BwdArgs a{};
  BwdMaps maps;
  if ((rc = bwd_setup(a, maps, kBF16, contiguous_inputs(q, k, v, dO, H, N, d), B, H, N, d, causal, scale)) !=
      EXATTN_OK)
    return rc;
  a.lse = lse;
  a.D = const_cast<float*>(D);
  a.dk = dk;
  a.sdk = contiguous(H, N, d);
  a.dv = dv;
  a.sdv = a.sdk;
  return launch_bwd_dkdv(a, static_cast<cudaStream_t>(stream)) == cudaSuccess ? EXATTN_OK : EXATTN_ERR_CUDA;
}

extern "C" int attn_bwd_dq(const void* q, const void* k, const void* v, const void* dO, const float* lse,
                           const float* D, void* dq, int B, int H, int N, int d, int causal, float scale,
                           void* stream) {
  if (!q || !k || !v || !dO || !lse || !D || !dq) return EXATTN_ERR_NULL;
  int rc = check_common(B, H, N, d, scale);
  if (rc != EXATTN_OK) return rc;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(dO, 16) || !aligned(dq, 16) ||
      !aligned(lse, 4) || !aligned(D, 4))
    return EXATTN_ERR_ALIGN;
  BwdArgs a{};
  BwdMaps maps;
  if ((rc = bwd_setup(a, maps, kBF16, contiguous_inputs(q, k, v, dO, H, N, d), B, H, N, d, causal, scale)) !=
      EXATTN_OK)
    return rc;
  a.lse = lse;
  a.D = const_cast<float*>(D);
  a.dq = dq;
  a.sdq = contiguous(H, N, d);
  return launch_bwd_dq(a, static_cast<cudaStream_t>(stream)) == cudaSuccess ? EXATTN_OK : EXATTN_ERR_CUDA;
}

extern "C" int attn_bwd_d_and_dq(const void* q, const void* k, const void* v, const void* o, const void* dO,
                                 const float* lse, float* D, void* dq, int B, int H, int N, int d, int causal,
                                 float scale, void* stream) {
  if (!q || !k || !v || !o || !dO || !lse || !D || !dq) return EXATTN_ERR_NULL;
  int rc = check_common(B, H, N, d, scale);
  if (rc != EXATTN_OK) return rc;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) || !aligned(dO, 16) ||
      !aligned(dq, 16) || !aligned(lse, 4) || !aligned(D, 4))
    return EXATTN_ERR_ALIGN;
  BwdArgs a{};
  BwdMaps maps;
  if ((rc = bwd_setup(a, maps, kBF16, contiguous_inputs(q, k, v, dO, H, N, d), B, H, N, d, causal, scale)) !=
      EXATTN_OK)
    return rc;
  a.o = o;
  a.so = contiguous(H, N, d);
  a.dO = dO;
  a.sdo = a.so;
  a.lse = lse;
  a.D = D;
  a.dq_computes_D = true;
  a.dq = dq;
  a.sdq = a.so;
  return launch_bwd_dq(a, static_cast<cudaStream_t>(stream)) == cudaSuccess ? EXATTN_OK : EXATTN_ERR_CUDA;
}

extern "C" int attn_bwd(const void* q, const void* k, const void* v, const void* o, const void* dO, const float* lse,
                        void* dq, void* dk, void* dv, int B, int H, int N, int d, int causal, float scale,
                        void* workspace, size_t workspace_bytes, void* stream) {
  if (!q || !k || !v || !o || !dO || !lse || !dq || !dk || !dv) return EXATTN_ERR_NULL;
  int rc = check_common(B, H, N, d, scale);
  if (rc != EXATTN_OK) return rc;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) || !aligned(dO, 16) ||
      !aligned(dq, 16) || !aligned(dk, 16) || !aligned(dv, 16) || !aligned(lse, 4))
    return EXATTN_ERR_ALIGN;
  if (!workspace || workspace_bytes < attn_bwd_workspace_size(B, H, N, d, causal)) return EXATTN_ERR_WORKSPACE;
  if (!aligned(workspace, 16)) return EXATTN_ERR_ALIGN;
  const Strides c = contiguous(H, N, d);
  return bwd_impl(kBF16, contiguous_inputs(q, k, v, dO, H, N, d), o, c, c, lse, dq, c, dk, c, dv, c, B, H, N, d,
                  causal, 0, scale, workspace, stream);
}

extern "C" int attn_bwd_ex(int dtype, const void* q, exattn_strides sq, const void* k, exattn_strides sk,
                           const void* v, exattn_strides sv, const void* o, exattn_strides so, const void* dO,
                           exattn_strides sdo, const float* lse, void* dq, exattn_strides sdq, void* dk,
                           exattn_strides sdk, void* dv, exattn_strides sdv, int B, int H, int N, int d, int causal,
                           int window, float scale, void* workspace, size_t workspace_bytes, void* stream) {
  if (!q || !k || !v || !o || !dO || !lse || !dq || !dk || !dv) return EXATTN_ERR_NULL;
  if (dtype != EXATTN_DTYPE_BF16 && dtype != EXATTN_DTYPE_F16) return EXATTN_ERR_UNSUPPORTED;
  int rc = check_common(B, H, N, d, scale);
  if (rc != EXATTN_OK) return rc;
  if (window < 0) return EXATTN_ERR_VALUE;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) || !aligned(dO, 16) ||
      !aligned(dq, 16) || !aligned(dk, 16) || !aligned(dv, 16) || !aligned(lse, 4))
    return EXATTN_ERR_ALIGN;
  const exattn_strides* all[8] = {&sq, &sk, &sv, &so, &sdo, &sdq, &sdk, &sdv};
  for (const exattn_strides* s : all)
    if ((rc = check_strides(*s, B, H, N)) != EXATTN_OK) return rc;
  if (!workspace || workspace_bytes < attn_bwd_workspace_size(B, H, N, d, causal)) return EXATTN_ERR_WORKSPACE;
  if (!aligned(workspace, 16)) return EXATTN_ERR_ALIGN;
  const BwdInputs in{{q, k, v, dO}, {to_strides(sq), to_strides(sk), to_strides(sv), to_strides(sdo)}};
  return bwd_impl(dtype == EXATTN_DTYPE_F16 ? kF16 : kBF16, in, o, to_strides(so), to_strides(sdo), lse, dq,
                  to_strides(sdq), dk, to_strides(sdk), dv, to_strides(sdv), B, H, N, d, causal, window, scale,
                  workspace, stream);
}

extern "C" int attn_bwd_o32(int dtype, const void* q, exattn_strides sq, const void* k, exattn_strides sk,
                            const void* v, exattn_strides sv, const float* o32, const void* dO, exattn_strides sdo,
                            const float* lse, void* dq, exattn_strides sdq, void* dk, exattn_strides sdk, void* dv,
                            exattn_strides sdv, int B, int H, int N, int d, int causal, int window, float scale,
                            void* workspace, size_t workspace_bytes, void* stream) {
  if (!q || !k || !v || !o32 || !dO || !lse || !dq || !dk || !dv) return EXATTN_ERR_NULL;
  if (dtype != EXATTN_DTYPE_BF16 && dtype != EXATTN_DTYPE_F16) return EXATTN_ERR_UNSUPPORTED;
  int rc = check_common(B, H, N, d, scale);
  if (rc != EXATTN_OK) return rc;
  if (window < 0) return EXATTN_ERR_VALUE;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o32, 16) || !aligned(dO, 16) ||
      !aligned(dq, 16) || !aligned(dk, 16) || !aligned(dv, 16) || !aligned(lse, 4))
    return EXATTN_ERR_ALIGN;
  const exattn_strides* all[7] = {&sq, &sk, &sv, &sdo, &sdq, &sdk, &sdv};
  for (const exattn_strides* s : all)
    if ((rc = check_strides(*s, B, H, N)) != EXATTN_OK) return rc;
  if (!workspace || workspace_bytes < attn_bwd_workspace_size(B, H, N, d, causal)) return EXATTN_ERR_WORKSPACE;
  if (!aligned(workspace, 16)) return EXATTN_ERR_ALIGN;
  const BwdInputs in{{q, k, v, dO}, {to_strides(sq), to_strides(sk), to_strides(sv), to_strides(sdo)}};
  const Strides c = contiguous(H, N, d);  // o32's layout (O itself is not read)
  return bwd_impl(dtype == EXATTN_DTYPE_F16 ? kF16 : kBF16, in, nullptr, c, to_strides(sdo), lse, dq, to_strides(sdq),
                  dk, to_strides(sdk), dv, to_strides(sdv), B, H, N, d, causal, window, scale, workspace, stream,
                  SeqView{nullptr, 0}, o32);
}

namespace {

// Shared checks of the packed variable-length calls.
int check_varlen(const int* cu_seqlens, int B, int H, int max_seqlen, int total, int d, float scale, int window) {
  if (!cu_seqlens) return EXATTN_ERR_NULL;
  if (!aligned(cu_seqlens, 4)) return EXATTN_ERR_ALIGN;
  if (total < 1 || static_cast<long long>(H) * total >= (1ll << 31)) return EXATTN_ERR_SHAPE;
  if (window < 0) return EXATTN_ERR_VALUE;
  return check_common(B, H, max_seqlen, d, scale);
}

}  // namespace

extern "C" int attn_fwd_varlen(int dtype, const void* q, exattn_strides sq, const void* k, exattn_strides sk,
                               const void* v, exattn_strides sv, void* o, exattn_strides so, float* lse,
                               const int* cu_seqlens, int B, int H, int max_seqlen, int total, int d, int causal,
                               int window, float scale, void* stream) {
  if (!q || !k || !v || !o || !lse) return EXATTN_ERR_NULL;
  if (dtype != EXATTN_DTYPE_BF16 && dtype != EXATTN_DTYPE_F16) return EXATTN_ERR_UNSUPPORTED;
  int rc = check_varlen(cu_seqlens, B, H, max_seqlen, total, d, scale, window);
  if (rc != EXATTN_OK) return rc;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) || !aligned(lse, 4))
    return EXATTN_ERR_ALIGN;
  const exattn_strides* all[4] = {&sq, &sk, &sv, &so};
  for (const exattn_strides* s : all)
    if ((rc = check_strides(*s, 1, H, total)) != EXATTN_OK) return rc;
  return fwd_impl(dtype == EXATTN_DTYPE_F16 ? kF16 : kBF16, q, to_strides(sq), k, to_strides(sk), v, to_strides(sv),
                  o, to_strides(so), lse, B, H, max_seqlen, d, causal, window, scale, stream,
                  SeqView{cu_seqlens, total});
}

extern "C" int attn_bwd_varlen(int dtype, const void* q, exattn_strides sq, const void* k, exattn_strides sk,
                               const void* v, exattn_strides sv, const void* o, exattn_strides so, const void* dO,
                               exattn_strides sdo, const float* lse, void* dq, exattn_strides sdq, void* dk,
                               exattn_strides sdk, void* dv, exattn_strides sdv, const int* cu_seqlens, int B, int H,
                               int max_seqlen, int total, int d, int causal, int window, float scale,
                               void* workspace, size_t workspace_bytes, void* stream) {
  if (!q || !k || !v || !o || !dO || !lse || !dq || !dk || !dv) return EXATTN_ERR_NULL;
  if (dtype != EXATTN_DTYPE_BF16 && dtype != EXATTN_DTYPE_F16) return EXATTN_ERR_UNSUPPORTED;
  int rc = check_varlen(cu_seqlens, B, H, max_seqlen, total, d, scale, window);
  if (rc != EXATTN_OK) return rc;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) || !aligned(dO, 16) ||
      !aligned(dq, 16) || !aligned(dk, 16) || !aligned(dv, 16) || !aligned(lse, 4))
    return EXATTN_ERR_ALIGN;
  const exattn_strides* all[8] = {&sq, &sk, &sv, &so, &sdo, &sdq, &sdk, &sdv};
  for (const exattn_strides* s : all)
    if ((rc = check_strides(*s, 1, H, total)) != EXATTN_OK) return rc;
  if (!workspace || workspace_bytes < attn_bwd_workspace_size(1, H, total, d, causal)) return EXATTN_ERR_WORKSPACE;
  if (!aligned(workspace, 16)) return EXATTN_ERR_ALIGN;
  const BwdInputs in{{q, k, v, dO}, {to_strides(sq), to_strides(sk), to_strides(sv), to_strides(sdo)}};
  return bwd_impl(dtype == EXATTN_DTYPE_F16 ? kF16 : kBF16, in, o, to_strides(so), to_strides(sdo), lse, dq,
                  to_strides(sdq), dk, to_strides(sdk), dv, to_strides(sdv), B, H, max_seqlen, d, causal, window,
                  scale, workspace, stream, SeqView{cu_seqlens, total});
}

namespace {

// Key splits of a decode-shaped forward (pick_splits below), no empty split.
struct DecodePlan {
  int n_splits, tiles_per_split, nq_pad;
  size_t o_bytes, lse_bytes, total_bytes;
};

// Key splits for a grid of `units` CTAs per split level (one per (batch,
// head), or per query-tile pair and (batch, head)) over nkt key tiles: the
// count whose grid finishes first when every CTA costs its key tiles plus
// a fixed set-up and epilogue of about three tiles' worth and the CTAs run
// in waves of one per SM (both kernels hold most of an SM's shared memory).
// A last wave that is nearly empty costs a whole CTA time, so a count that
// fills one wave with longer CTAs beats one that spills a few CTAs into a
// second.  At most about two waves of CTAs: beyond that every SM already
// streams keys and more splits add only set-up costs.  At most max_splits
// splits; ties go to fewer splits (less workspace, a smaller merge).
long long pick_splits(long long units, long long nkt, long long max_splits) {
  constexpr long long kSMs = 152, kFixedTiles = 3;
  max_splits = std::min(max_splits, 2 * kSMs / std::max(1ll, units));
  max_splits = std::max(1ll, std::min({max_splits, nkt, static_cast<long long>(kMaxSplits)}));
  long long best = 1, best_cost = -1;
  for (long long s = 1; s <= max_splits; ++s) {
    const long long tps = (nkt + s - 1) / s, used = (nkt + tps - 1) / tps;
    const long long cost = ((units * used + kSMs - 1) / kSMs) * (kFixedTiles + tps);
    if (best_cost < 0 || cost < best_cost) {
      best_cost = cost;
      best = used;
    }
  }
  return best;
}

DecodePlan decode_plan(int B, int H, int Nq, int Nk, int d) {
  const long long nkt = (Nk + 127) / 128;
  const long long bh = static_cast<long long>(B) * H;
  long long splits;
  int nq_pad;
  if (Nq <= kDecodeMaxQ && d == 128) {
    // The decode kernel: one CTA per (batch, head) and key split, at least
    // four key tiles per split where the keys allow it.
    splits = pick_splits(bh, nkt, nkt / 4);
    nq_pad = kDecodeQCols;
  } else {
    // The forward kernel with its keys split: pairs of 128-row query tiles,
    // at least two key tiles per split.
    const int n_pairs = (Nq + 255) / 256;
    splits = pick_splits(static_cast<long long>(n_pairs) * bh, nkt, nkt / 2);
    nq_pad = n_pairs * 256;
  }
  const long long tps = (nkt + splits - 1) / splits;
  splits = (nkt + tps - 1) / tps;
  DecodePlan p{static_cast<int>(splits), static_cast<int>(tps), nq_pad, 0, 0, 0};
  if (p.n_splits > 1) {
    const size_t rows = static_cast<size_t>(p.n_splits) * B * H * p.nq_pad;
    p.o_bytes = (rows * d * sizeof(float) + 255) & ~size_t(255);
    p.lse_bytes = (rows * sizeof(float) + 255) & ~size_t(255);
    p.total_bytes = p.o_bytes + 2 * p.lse_bytes;
  }
  return p;
}

int check_decode(int B, int H, int Nq, int Nk, int d, int causal, int window, float scale) {
  if (Nq < 1 || Nk < 1) return EXATTN_ERR_SHAPE;
  if ((causal || window > 0) && Nq > Nk) return EXATTN_ERR_SHAPE;  // a query with no key at or before it
  if (window < 0) return EXATTN_ERR_VALUE;
  if (static_cast<long long>(B) * H * Nk >= (1ll << 31)) return EXATTN_ERR_SHAPE;
  return check_common(B, H, Nq, d, scale);
}

}  // namespace

extern "C" size_t attn_fwd_decode_workspace_size(int B, int H, int Nq, int Nk, int d) {
  if (check_decode(B, H, Nq, Nk, d, 0, 0, 1.f) != EXATTN_OK) return 0;
  return decode_plan(B, H, Nq, Nk, d).total_bytes;
}

extern "C" int attn_fwd_decode(int dtype, const void* q, exattn_strides sq, const void* k, exattn_strides sk,
                               const void* v, exattn_strides sv, void* o, exattn_strides so, float* lse, int B,
                               int H, int Nq, int Nk, int d, int causal, int window, float scale, void* workspace,
                               size_t workspace_bytes, void* stream) {
  if (!q || !k || !v || !o || !lse) return EXATTN_ERR_NULL;
  if (dtype != EXATTN_DTYPE_BF16 && dtype != EXATTN_DTYPE_F16) return EXATTN_ERR_UNSUPPORTED;
  int rc = check_decode(B, H, Nq, Nk, d, causal, window, scale);
  if (rc != EXATTN_OK) return rc;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) || !aligned(lse, 4))
    return EXATTN_ERR_ALIGN;
  if ((rc = check_strides(sq, B, H, Nq)) != EXATTN_OK || (rc = check_strides(so, B, H, Nq)) != EXATTN_OK ||
      (rc = check_strides(sk, B, H, Nk)) != EXATTN_OK || (rc = check_strides(sv, B, H, Nk)) != EXATTN_OK)
    return rc;
  const DecodePlan plan = decode_plan(B, H, Nq, Nk, d);
  if (plan.total_bytes > 0) {
    if (!workspace || workspace_bytes < plan.total_bytes) return EXATTN_ERR_WORKSPACE;
    if (!aligned(workspace, 16)) return EXATTN_ERR_ALIGN;
  }
  int dev = 0;
  unsigned* err = nullptr;
  if ((rc = device_setup(&dev, &err)) != EXATTN_OK) return rc;
  const int dt = dtype == EXATTN_DTYPE_F16 ? kF16 : kBF16;
  const bool few_queries = Nq <= kDecodeMaxQ && d == 128;  // the decode kernel, else the forward with key splits
  CUtensorMap mq, mk, mv;
  if (!make_map(&mq, q, dt, B, H, Nq, d, to_strides(sq), few_queries ? kDecodeQCols : 128) ||
      !make_map(&mk, k, dt, B, H, Nk, d, to_strides(sk), 128) ||
      !make_map(&mv, v, dt, B, H, Nk, d, to_strides(sv), 128))
    return EXATTN_ERR_CUDA;
  FwdArgs a{};
  a.tm_q = &mq;
  a.tm_k = &mk;
  a.tm_v = &mv;
  a.o = o;
  a.so = to_strides(so);
  a.lse = lse;
  a.N = Nq;
  a.H = H;
  a.BH = B * H;
  a.d = d;
  a.causal = causal ? 1 : 0;
  a.dtype = dt;
  a.window = window;
  a.seq = SeqView{nullptr, 0};
  a.kv.nk = Nk;
  a.kv.n_splits = plan.n_splits;
  a.kv.tiles_per_split = plan.tiles_per_split;
  a.kv.nq_pad = plan.nq_pad;
  if (plan.n_splits > 1) {
    char* ws = static_cast<char*>(workspace);
    a.kv.part_o = reinterpret_cast<float*>(ws);
    a.kv.part_lse = reinterpret_cast<float*>(ws + plan.o_bytes);
    a.kv.part_lseb = reinterpret_cast<float*>(ws + plan.o_bytes + plan.lse_bytes);
  }
  a.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  a.err = err;
  a.device = dev;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  if ((few_queries ? launch_decode(a, st) : launch_fwd(a, st)) != cudaSuccess) return EXATTN_ERR_CUDA;
  if (plan.n_splits > 1 && launch_fwd_merge(a, st) != cudaSuccess) return EXATTN_ERR_CUDA;
  return EXATTN_OK;
}

extern "C" const char* exattn_status_string(int status) {
  switch (status) {
    case EXATTN_OK: return "ok";
    case EXATTN_ERR_NULL: return "a required pointer is NULL";
    case EXATTN_ERR_SHAPE: return "B, H or N out of range";
    case EXATTN_ERR_ALIGN: return "a pointer is misaligned (bf16 tensors and workspace need 16 bytes, lse 4)";
    case EXATTN_ERR_UNSUPPORTED: return "head dimension d must be 64 or 128";
    case EXATTN_ERR_ARCH: return "the current device is not sm_103 (GB300)";
    case EXATTN_ERR_WORKSPACE: return "workspace is NULL or smaller than attn_bwd_workspace_size()";
    case EXATTN_ERR_CUDA: return "a CUDA call or kernel launch failed";
    case EXATTN_ERR_TIMEOUT: return "a kernel's bounded internal wait gave up; outputs are invalid";
    case EXATTN_ERR_VALUE: return "scale must be finite and positive";
    default: return "unknown exattn status";
  }
}

extern "C" int exattn_device_error(void) {
  int dev = 0;
  unsigned* err = nullptr;
  int rc = device_setup(&dev, &err);
  if (rc != EXATTN_OK) return rc;
  if (note_cuda(cudaDeviceSynchronize(), "cudaDeviceSynchronize") != cudaSuccess) return EXATTN_ERR_CUDA;
  unsigned v = 0;
  if (note_cuda(cudaMemcpyFromSymbol(&v, g_err_word, sizeof(v)), "cudaMemcpyFromSymbol") != cudaSuccess)
    return EXATTN_ERR_CUDA;
  if (v != 0) {
    const unsigned zero = 0;
    if (note_cuda(cudaMemcpyToSymbol(g_err_word, &zero, sizeof(zero)), "cudaMemcpyToSymbol") != cudaSuccess)
      return EXATTN_ERR_CUDA;
    return EXATTN_ERR_TIMEOUT;
  }
  return EXATTN_OK;
}

extern "C" int exattn_device_error_poll(unsigned* host_dst, void* stream) {
  if (!host_dst) return EXATTN_ERR_NULL;
  int dev = 0;
  unsigned* err = nullptr;
  int rc = device_setup(&dev, &err);
  if (rc != EXATTN_OK) return rc;
  return note_cuda(cudaMemcpyAsync(host_dst, err, sizeof(unsigned), cudaMemcpyDeviceToHost,
                                   static_cast<cudaStream_t>(stream)),
                   "cudaMemcpyAsync") == cudaSuccess
             ? EXATTN_OK
             : EXATTN_ERR_CUDA;
}

extern "C" int exattn_watchdog_selftest(unsigned timeout_us, void* stream) {
  if (timeout_us < 1 || timeout_us > 1000000) return EXATTN_ERR_VALUE;
  int dev = 0;
  unsigned* err = nullptr;
  int rc = device_setup(&dev, &err);
  if (rc != EXATTN_OK) return rc;
  watchdog_selftest_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(1000ull * timeout_us, err);
  return note_cuda(cudaGetLastError(), "watchdog self-test kernel launch") == cudaSuccess ? EXATTN_OK : EXATTN_ERR_CUDA;
}

extern "C" const char* exattn_last_cuda_error(void) {
  if (!t_fail_call) return "";
  if (t_fail_driver)
    std::snprintf(t_fail_text, sizeof(t_fail_text), "%s: CUresult %d", t_fail_call, t_fail_code);
  else
    std::snprintf(t_fail_text, sizeof(t_fail_text), "%s: %s (%d)", t_fail_call,
                  cudaGetErrorName(static_cast<cudaError_t>(t_fail_code)), t_fail_code);
  return t_fail_text;
}

extern "C" int exattn_version(void) { return 202; }  // 0.2.2: fp32-O calls, exattn_last_cuda_error
