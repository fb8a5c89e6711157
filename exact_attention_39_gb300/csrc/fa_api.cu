// fa_api.cu -- host side of the C ABI declared in include/fa.h: argument
// checks, TMA tensor-map encoding, kernel launch, device status word.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "fa.h"
#include "fa_fwd_kernel.cuh"

namespace fa {

// Per-device status word: bit kStatusTimeout is set by a kernel whose bounded
// wait ran out.  Read and cleared by fa_last_device_error().
__device__ unsigned g_device_status = 0u;

namespace {

constexpr int kMaxDevices = 64;
constexpr unsigned long long kTimeoutNs = 2000000000ull;   // 2 s per wait

std::mutex g_mutex;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
bool g_dev_ready[kMaxDevices] = {};
unsigned *g_status_ptr[kMaxDevices] = {};

template <int D, bool BF16>
void *kernel_ptr() {
  return reinterpret_cast<void *>(&fa_fwd_kernel<D, BF16>);
}

// One-time, per-process and per-device set-up: the driver's tensor-map
// encoder, the kernels' shared-memory opt-in, the status word's address.
fa_status ensure_ready(int dev) {
  std::lock_guard<std::mutex> lock(g_mutex);
  if (!g_encode) {
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                         cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fn)
      return FA_ERR_CUDA;
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  if (dev < 0 || dev >= kMaxDevices) return FA_ERR_CUDA;
  if (g_dev_ready[dev]) return FA_OK;
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return FA_ERR_CUDA;
  if (major != 10 || minor != 3) return FA_ERR_CUDA;   // built for sm_103a only
  const void *kernels[4] = {kernel_ptr<64, false>(), kernel_ptr<64, true>(),
                            kernel_ptr<128, false>(), kernel_ptr<128, true>()};
  const int smem[4] = {Layout<64>::kAlloc, Layout<64>::kAlloc,
                       Layout<128>::kAlloc, Layout<128>::kAlloc};
  for (int t = 0; t < 4; ++t)
    if (cudaFuncSetAttribute(kernels[t], cudaFuncAttributeMaxDynamicSharedMemorySize,
                             smem[t]) != cudaSuccess)
      return FA_ERR_CUDA;
  void *addr = nullptr;
  if (cudaGetSymbolAddress(&addr, g_device_status) != cudaSuccess || !addr)
    return FA_ERR_CUDA;
  g_status_ptr[dev] = static_cast<unsigned *>(addr);
  g_dev_ready[dev] = true;
  return FA_OK;
}

// [BH, rows, d] tensor viewed by TMA as a 3-D box grid of 64 x 128 x 1
// elements (128-byte rows, 128-byte swizzle).  Rows past `rows` within a
// head read as zero.
bool encode_map(CUtensorMap *map, const void *base, bool bf16, int d, int rows,
                long long bh) {
  cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)rows, (cuuint64_t)bh};
  cuuint64_t strides[2] = {(cuuint64_t)d * 2u, (cuuint64_t)d * 2u * (cuuint64_t)rows};
  cuuint32_t box[3] = {64u, 128u, 1u};
  cuuint32_t estr[3] = {1u, 1u, 1u};
  CUresult r = g_encode(map,
                        bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                             : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                        3, const_cast<void *>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

template <int D, bool BF16>
cudaError_t launch(const CUtensorMap &mq, const CUtensorMap &mk,
                   const CUtensorMap &mv, const FwdParams &p, unsigned grid,
                   cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = Layout<D>::kAlloc;
  cfg.stream = stream;
  return cudaLaunchKernelEx(&cfg, fa_fwd_kernel<D, BF16>, mq, mk, mv, p);
}

bool aligned(const void *p, uintptr_t a) {
  return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0;
}

}  // namespace
}  // namespace fa

extern "C" {

fa_status fa_fwd_qk(const void *q, const void *k, const void *v, void *o,
                    float *lse, int B, int H, int Nq, int Nk, int d, int causal,
                    float scale, fa_dtype dtype, fa_stream_t stream) {
  using namespace fa;
  if (B < 0 || H < 0 || Nq < 0 || Nk < 0) return FA_ERR_SHAPE;
  if (d != 64 && d != 128) return FA_ERR_HEADDIM;
  if (dtype != FA_FP16 && dtype != FA_BF16) return FA_ERR_DTYPE;
  if (!std::isfinite(scale) || !(scale > 0.f)) return FA_ERR_SCALE;
  if (B == 0 || H == 0 || Nq == 0) return FA_OK;   // empty problem
  const long long bh = (long long)B * (long long)H;
  const long long units = ((long long)Nq + kRowsPerCta - 1) / kRowsPerCta;
  if (bh > (1ll << 31) - 1 || bh * units > (1ll << 31) - 1) return FA_ERR_SHAPE;
  if (!q || !o || !lse || (Nk > 0 && (!k || !v))) return FA_ERR_NULL;
  if (!aligned(q, 16) || !aligned(o, 16) || !aligned(lse, 4) ||
      (Nk > 0 && (!aligned(k, 16) || !aligned(v, 16))))
    return FA_ERR_ALIGN;

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_CUDA;
  fa_status st = ensure_ready(dev);
  if (st != FA_OK) return st;

  const bool bf16 = dtype == FA_BF16;
  // With no keys the kernel loads nothing from K or V; their maps are
  // built over q only to be well formed.
  const void *kb = Nk > 0 ? k : q, *vb = Nk > 0 ? v : q;
  const int nk_map = Nk > 0 ? Nk : Nq;
  CUtensorMap mq, mk, mv;
  if (!encode_map(&mq, q, bf16, d, Nq, bh) || !encode_map(&mk, kb, bf16, d, nk_map, bh) ||
      !encode_map(&mv, vb, bf16, d, nk_map, bh))
    return FA_ERR_CUDA;

  FwdParams p;
  p.o = o;
  p.lse = lse;
  p.Nq = Nq;
  p.Nk = Nk;
  p.n_units = (int)units;
  p.causal = causal ? 1 : 0;
  p.c = (float)((double)scale * 1.4426950408889634);
  p.timeout_ns = kTimeoutNs;
  p.status = g_status_ptr[dev];

  const unsigned grid = (unsigned)(bh * units);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t err;
  if (d == 64)
    err = bf16 ? launch<64, true>(mq, mk, mv, p, grid, s)
               : launch<64, false>(mq, mk, mv, p, grid, s);
  else
    err = bf16 ? launch<128, true>(mq, mk, mv, p, grid, s)
               : launch<128, false>(mq, mk, mv, p, grid, s);
  return err == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

fa_status fa_fwd(const void *q, const void *k, const void *v, void *o,
                 float *lse, int B, int H, int N, int d, int causal,
                 float scale, fa_dtype dtype, fa_stream_t stream) {
  if (N < 0) return FA_ERR_SHAPE;
  return fa_fwd_qk(q, k, v, o, lse, B, H, N, N, d, causal, scale, dtype, stream);
}

const char *fa_status_string(fa_status status) {
  switch (status) {
    case FA_OK: return "ok";
    case FA_ERR_NULL: return "a required pointer is NULL";
    case FA_ERR_SHAPE: return "B, H or N is negative or too large";
    case FA_ERR_HEADDIM: return "head dimension must be 64 or 128";
    case FA_ERR_DTYPE: return "dtype must be FA_FP16 or FA_BF16";
    case FA_ERR_ALIGN: return "q/k/v/o must be 16-byte aligned and lse 4-byte aligned";
    case FA_ERR_SCALE: return "scale must be finite and positive";
    case FA_ERR_CUDA: return "CUDA error (call failed, or device is not sm_103)";
    case FA_ERR_DEVICE_TIMEOUT: return "a bounded on-device wait timed out";
  }
  return "unknown status";
}

fa_status fa_last_device_error(fa_stream_t stream) {
  using namespace fa;
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return FA_ERR_CUDA;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_CUDA;
  fa_status st = ensure_ready(dev);
  if (st != FA_OK) return st;
  unsigned word = 0;
  if (cudaMemcpyFromSymbol(&word, g_device_status, sizeof(word)) != cudaSuccess)
    return FA_ERR_CUDA;
  if (word == 0) return FA_OK;
  const unsigned zero = 0;
  if (cudaMemcpyToSymbol(g_device_status, &zero, sizeof(zero)) != cudaSuccess)
    return FA_ERR_CUDA;
  return FA_ERR_DEVICE_TIMEOUT;
}

int fa_version(void) { return 100; }

}  // extern "C"
