// api.cu -- the C ABI of libexattn.so (declared in include/exattn.h):
// argument validation, per-device set-up, TMA tensor-map encoding and kernel
// launches.  No device memory is allocated here and nothing synchronises
// except exattn_device_error().
#include <cmath>
#include <cstdint>
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

constexpr int kMaxDevices = 64;

struct DeviceState {
  bool ready = false;
  int status = EXATTN_OK;  // EXATTN_OK, EXATTN_ERR_ARCH or EXATTN_ERR_CUDA once set up
  unsigned* err = nullptr;
};

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];
EncodeTiledFn g_encode = nullptr;

struct AttrKey {
  const void* fn;
  int device;
};
AttrKey g_attr_done[256];
int g_attr_count = 0;

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// Arch check, watchdog address and the tensor-map encoder, once per device.
int device_setup(int* dev_out, unsigned** err_out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return EXATTN_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return EXATTN_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceState& st = g_dev[dev];
  if (!st.ready) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
      return EXATTN_ERR_CUDA;
    }
    if (major != 10 || minor != 3) {
      st.status = EXATTN_ERR_ARCH;
    } else {
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, g_err_word) != cudaSuccess) return EXATTN_ERR_CUDA;
      st.err = static_cast<unsigned*>(p);
      if (!g_encode) {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess || !fn) {
          return EXATTN_ERR_CUDA;
        }
        g_encode = reinterpret_cast<EncodeTiledFn>(fn);
      }
      st.status = EXATTN_OK;
    }
    st.ready = true;
  }
  *dev_out = dev;
  *err_out = st.err;
  return st.status;
}

// [B*H, N, d] bf16, d contiguous; box = 64 columns (128 bytes) x box_rows rows x 1.
bool make_map(CUtensorMap* m, const void* base, int BH, int N, int d, int box_rows) {
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(BH)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2, static_cast<cuuint64_t>(N) * d * 2};
  const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(box_rows), 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int check_common(int B, int H, int N, int d, float scale) {
  if (B < 1 || H < 1 || N < 1) return EXATTN_ERR_SHAPE;
  if (static_cast<long long>(B) * H * N >= (1ll << 31)) return EXATTN_ERR_SHAPE;
  if (static_cast<long long>(B) * H >= (1ll << 24)) return EXATTN_ERR_SHAPE;
  if (d != 64 && d != 128) return EXATTN_ERR_UNSUPPORTED;
  if (!std::isfinite(scale) || !(scale > 0.f)) return EXATTN_ERR_VALUE;
  return EXATTN_OK;
}

}  // namespace

cudaError_t ensure_smem_attr(const void* kernel, int bytes, int device) {
  std::lock_guard<std::mutex> lk(g_mu);
  for (int i = 0; i < g_attr_count; ++i)
    if (g_attr_done[i].fn == kernel && g_attr_done[i].device == device) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) return e;
  if (g_attr_count < 256) g_attr_done[g_attr_count++] = AttrKey{kernel, device};
  return cudaSuccess;
}

}  // namespace exattn

using namespace exattn;

extern "C" int attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int d,
                        int causal, float scale, void* stream) {
  if (!q || !k || !v || !o || !lse) return EXATTN_ERR_NULL;
  int rc = check_common(B, H, N, d, scale);
  if (rc != EXATTN_OK) return rc;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) || !aligned(lse, 4))
    return EXATTN_ERR_ALIGN;
  int dev = 0;
  unsigned* err = nullptr;
  if ((rc = device_setup(&dev, &err)) != EXATTN_OK) return rc;
  const int BH = B * H;
  CUtensorMap mq, mk, mv;
  if (!make_map(&mq, q, BH, N, d, 128) || !make_map(&mk, k, BH, N, d, 128) || !make_map(&mv, v, BH, N, d, 128))
    return EXATTN_ERR_CUDA;
  FwdArgs a;
  a.tm_q = &mq;
  a.tm_k = &mk;
  a.tm_v = &mv;
  a.o = o;
  a.lse = lse;
  a.N = N;
  a.BH = BH;
  a.d = d;
  a.causal = causal ? 1 : 0;
  a.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  a.err = err;
  a.device = dev;
  return launch_fwd(a, static_cast<cudaStream_t>(stream)) == cudaSuccess ? EXATTN_OK : EXATTN_ERR_CUDA;
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
  CUtensorMap m[8];
};

int bwd_setup(BwdArgs& a, BwdMaps& maps, const void* q, const void* k, const void* v, const void* dO, int B, int H,
              int N, int d, int causal, float scale) {
  int dev = 0;
  unsigned* err = nullptr;
  int rc = device_setup(&dev, &err);
  if (rc != EXATTN_OK) return rc;
  const int BH = B * H;
  const void* src[4] = {q, k, v, dO};
  for (int i = 0; i < 4; ++i) {
    if (!src[i]) continue;
    if (!make_map(&maps.m[i], src[i], BH, N, d, 128) || !make_map(&maps.m[4 + i], src[i], BH, N, d, 64))
      return EXATTN_ERR_CUDA;
  }
  a.tm_q128 = &maps.m[0];
  a.tm_k128 = &maps.m[1];
  a.tm_v128 = &maps.m[2];
  a.tm_do128 = &maps.m[3];
  a.tm_q64 = &maps.m[4];
  a.tm_k64 = &maps.m[5];
  a.tm_v64 = &maps.m[6];
  a.tm_do64 = &maps.m[7];
  a.N = N;
  a.BH = BH;
  a.d = d;
  a.causal = causal ? 1 : 0;
  a.scale = scale;
  a.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  a.err = err;
  a.device = dev;
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
  if ((rc = bwd_setup(a, maps, nullptr, nullptr, nullptr, nullptr, B, H, N, d, 0, 1.f)) != EXATTN_OK) return rc;
  a.o = o;
  a.dO = dO;
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
  if ((rc = bwd_setup(a, maps, q, k, v, dO, B, H, N, d, causal, scale)) != EXATTN_OK) return rc;
  a.lse = lse;
  a.D = const_cast<float*>(D);
  a.dk = dk;
  a.dv = dv;
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
  if ((rc = bwd_setup(a, maps, q, k, v, dO, B, H, N, d, causal, scale)) != EXATTN_OK) return rc;
  a.lse = lse;
  a.D = const_cast<float*>(D);
  a.dq = dq;
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
  BwdArgs a{};
  BwdMaps maps;
  if ((rc = bwd_setup(a, maps, q, k, v, dO, B, H, N, d, causal, scale)) != EXATTN_OK) return rc;
  a.o = o;
  a.dO = dO;
  a.lse = lse;
  a.dq = dq;
  a.dk = dk;
  a.dv = dv;
  a.D = static_cast<float*>(workspace);
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (launch_bwd_prep(a, st) != cudaSuccess) return EXATTN_ERR_CUDA;
  if (launch_bwd_dkdv(a, st) != cudaSuccess) return EXATTN_ERR_CUDA;
  if (launch_bwd_dq(a, st) != cudaSuccess) return EXATTN_ERR_CUDA;
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
  if (cudaDeviceSynchronize() != cudaSuccess) return EXATTN_ERR_CUDA;
  unsigned v = 0;
  if (cudaMemcpyFromSymbol(&v, g_err_word, sizeof(v)) != cudaSuccess) return EXATTN_ERR_CUDA;
  if (v != 0) {
    const unsigned zero = 0;
    if (cudaMemcpyToSymbol(g_err_word, &zero, sizeof(zero)) != cudaSuccess) return EXATTN_ERR_CUDA;
    return EXATTN_ERR_TIMEOUT;
  }
  return EXATTN_OK;
}

extern "C" int exattn_watchdog_selftest(unsigned timeout_us, void* stream) {
  if (timeout_us < 1 || timeout_us > 1000000) return EXATTN_ERR_VALUE;
  int dev = 0;
  unsigned* err = nullptr;
  int rc = device_setup(&dev, &err);
  if (rc != EXATTN_OK) return rc;
  watchdog_selftest_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(1000ull * timeout_us, err);
  return cudaGetLastError() == cudaSuccess ? EXATTN_OK : EXATTN_ERR_CUDA;
}

extern "C" int exattn_version(void) { return 100; }
