// fa_api.cu -- host side of the C ABI declared in include/fa.h: argument
// checks, TMA tensor-map encoding, kernel launch, device status word.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "fa.h"
#include "fa_selftest.h"
#include "fa_bwd_kernel.cuh"
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

template <int D, int T, int Q = 2, bool kSkip = false>
void *kernel_ptr() {
  return reinterpret_cast<void *>(&fa_fwd_kernel<D, T, Q, kSkip>);
}

// Key lengths up to which D = 64 runs one query tile per CTA, two CTAs per
// SM (CtaShape<1>), for 16-bit inputs.  Two resident CTAs overlap one's
// set-up, first loads, epilogue and exit with the other's key blocks, which a
// lone two-tile CTA leaves the SM idle for (about 5000 cycles a CTA, measured
// with a clock64 trace); in steady state the two-tile CTA's key block is
// about 7 % cheaper per query tile.  Measured against the two-tile shape at
// B8 H32 d64 bf16: N512 +10 %, N1024 +7 %, N2048 +5 %, N4096 +0.5 %
// (causal N2048 +3.5 %, N4096 +1 %), N8192 -3.5 % (causal -2 %).  e4m3
// inputs halve the tensor time of a block, so the overlap pays at every
// length (N4096 +6 %, N8192 +3 %, causal N8192 +4 %): they always take one
// tile.
constexpr int kOneTileMaxNk = 4096;

// One-time, per-process and per-device set-up: the CUDA driver's
// tensor-map encoder, the kernels' shared-memory opt-in, the status word's address.
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
  // Every forward instantiation the host launches, its shared memory, and
  // whether two of its CTAs share an SM (the one-tile shape, which needs the
  // whole carveout as shared memory).  The causal two-tile d = 64 kernels
  // (last argument true) skip tile 0's block past its diagonal.
  struct FwdKernel { const void *fn; int smem; bool two_per_sm; };
  const FwdKernel fwd_kernels[] = {
      {kernel_ptr<64, kF16>(), Layout<64, kF16>::kAlloc, false},
      {kernel_ptr<64, kBF16>(), Layout<64, kBF16>::kAlloc, false},
      {kernel_ptr<64, kF16, 2, true>(), Layout<64, kF16>::kAlloc, false},
      {kernel_ptr<64, kBF16, 2, true>(), Layout<64, kBF16>::kAlloc, false},
      {kernel_ptr<128, kF16>(), Layout<128, kF16>::kAlloc, false},
      {kernel_ptr<128, kBF16>(), Layout<128, kBF16>::kAlloc, false},
      {kernel_ptr<128, kE4M3>(), Layout<128, kE4M3>::kAlloc, false},
      {kernel_ptr<64, kF16, 1>(), Layout<64, kF16, 1>::kAlloc, true},
      {kernel_ptr<64, kBF16, 1>(), Layout<64, kBF16, 1>::kAlloc, true},
      {kernel_ptr<64, kE4M3, 1>(), Layout<64, kE4M3, 1>::kAlloc, true}};
  for (const FwdKernel &k : fwd_kernels) {
    if (cudaFuncSetAttribute(k.fn, cudaFuncAttributeMaxDynamicSharedMemorySize, k.smem) !=
        cudaSuccess)
      return FA_ERR_CUDA;
    if (k.two_per_sm && cudaFuncSetAttribute(k.fn, cudaFuncAttributePreferredSharedMemoryCarveout,
                                             100) != cudaSuccess)
      return FA_ERR_CUDA;
  }
  const void *bwd_kernels[8] = {
      reinterpret_cast<void *>(&fa_bwd_dq_kernel<64, kF16>),
      reinterpret_cast<void *>(&fa_bwd_dq_kernel<64, kBF16>),
      reinterpret_cast<void *>(&fa_bwd_dq_kernel<128, kF16>),
      reinterpret_cast<void *>(&fa_bwd_dq_kernel<128, kBF16>),
      reinterpret_cast<void *>(&fa_bwd_dkdv_kernel<64, kF16>),
      reinterpret_cast<void *>(&fa_bwd_dkdv_kernel<64, kBF16>),
      reinterpret_cast<void *>(&fa_bwd_dkdv_kernel<128, kF16>),
      reinterpret_cast<void *>(&fa_bwd_dkdv_kernel<128, kBF16>)};
  const int bwd_smem[8] = {BwdQLayout<64, kF16>::kAlloc, BwdQLayout<64, kBF16>::kAlloc,
                           BwdQLayout<128, kF16>::kAlloc, BwdQLayout<128, kBF16>::kAlloc,
                           BwdKVLayout<64, kF16>::kAlloc, BwdKVLayout<64, kBF16>::kAlloc,
                           BwdKVLayout<128, kF16>::kAlloc, BwdKVLayout<128, kBF16>::kAlloc};
  for (int t = 0; t < 8; ++t)
    if (cudaFuncSetAttribute(bwd_kernels[t], cudaFuncAttributeMaxDynamicSharedMemorySize,
                             bwd_smem[t]) != cudaSuccess)
      return FA_ERR_CUDA;
  void *addr = nullptr;
  if (cudaGetSymbolAddress(&addr, g_device_status) != cudaSuccess || !addr)
    return FA_ERR_CUDA;
  g_status_ptr[dev] = static_cast<unsigned *>(addr);
  g_dev_ready[dev] = true;
  return FA_OK;
}

// [BH, rows, d] tensor viewed by TMA as a 3-D box grid of (chunk width) x
// box_rows x 1 elements in the swizzle the kernel's layout names (box_rows:
// 128 for whole tiles, 64 for the backward's inner blocks).  Rows past
// `rows` within a head read as zero.
template <int D, int T>
bool encode_map_uncached(CUtensorMap *map, const void *base, int rows, long long bh,
                         int box_rows) {
  using L = Layout<D, T>;
  const cuuint64_t eb = (cuuint64_t)Elem<T>::kBytes;
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)rows, (cuuint64_t)bh};
  cuuint64_t strides[2] = {(cuuint64_t)D * eb, (cuuint64_t)D * eb * (cuuint64_t)rows};
  cuuint32_t box[3] = {(cuuint32_t)L::kChunkElems, (cuuint32_t)box_rows, 1u};
  cuuint32_t estr[3] = {1u, 1u, 1u};
  const CUtensorMapDataType dt = T == kF16    ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                 : T == kBF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                              : CU_TENSOR_MAP_DATA_TYPE_UINT8;
  CUresult r = g_encode(map, dt, 3, const_cast<void *>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE,
                        L::kSwz == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                                       : CU_TENSOR_MAP_SWIZZLE_64B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// A tensor map depends only on (base address, rows, heads, head dim, element
// type, box height), so the maps of recent calls are kept and reused: a call
// on the same buffers skips the driver's encoder.  Small and round-robin; a
// map is a plain 128-byte value (no driver object to release).
struct MapKey {
  const void *base;
  long long bh;
  int rows, d, t, box_rows;
  bool operator==(const MapKey &o) const {
    return base == o.base && bh == o.bh && rows == o.rows && d == o.d && t == o.t &&
           box_rows == o.box_rows;
  }
};
struct MapEntry {
  MapKey key;
  CUtensorMap map;
  bool valid;
};
constexpr int kMapCacheSize = 64;
MapEntry g_map_cache[kMapCacheSize] = {};
int g_map_next = 0;
std::mutex g_map_mutex;

template <int D, int T>
bool encode_map(CUtensorMap *map, const void *base, int rows, long long bh,
                int box_rows = kBM) {
  const MapKey key{base, bh, rows, D, T, box_rows};
  {
    std::lock_guard<std::mutex> lock(g_map_mutex);
    for (const MapEntry &e : g_map_cache)
      if (e.valid && e.key == key) {
        *map = e.map;
        return true;
      }
  }
  if (!encode_map_uncached<D, T>(map, base, rows, bh, box_rows)) return false;
  std::lock_guard<std::mutex> lock(g_map_mutex);
  MapEntry &e = g_map_cache[g_map_next];
  g_map_next = (g_map_next + 1) % kMapCacheSize;
  e.key = key;
  e.map = *map;
  e.valid = true;
  return true;
}

// Encodes the maps and launches one forward kernel.  With no keys the
// kernel loads nothing from K or V; their maps are built over q only to be
// well formed.
template <int D, int T, int Q>
fa_status run_shape(const CUtensorMap &mq, const CUtensorMap &mk, const CUtensorMap &mv,
                    FwdParams p, long long bh, cudaStream_t stream) {
  const long long units = ((long long)p.Nq + Q * kBM - 1) / (Q * kBM);
  if (bh * units > (1ll << 31) - 1) return FA_ERR_SHAPE;
  p.n_units = (int)units;
  // causal work order: heads per group, from the bytes of one head's K and V
  const long long kv_head = 2ll * p.Nk * D * Elem<T>::kBytes;
  long long group = kv_head > 0 ? kCausalGroupKVBytes / kv_head : kCausalMaxHeadGroup;
  group = std::min<long long>(std::max<long long>(group, 1), kCausalMaxHeadGroup);
  p.head_group = (int)std::min<long long>(group, bh);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(bh * units), 1, 1);
  cfg.blockDim = dim3(CtaShape<Q>::kThreads, 1, 1);
  cfg.dynamicSmemBytes = Layout<D, T, Q>::kAlloc;
  cfg.stream = stream;
  cudaError_t e;
  if constexpr (D == 64 && Q == 2) {
    // causal: tile 0 skips a block past its diagonal (its own instantiation)
    e = p.causal ? cudaLaunchKernelEx(&cfg, fa_fwd_kernel<D, T, Q, true>, mq, mk, mv, p)
                 : cudaLaunchKernelEx(&cfg, fa_fwd_kernel<D, T, Q, false>, mq, mk, mv, p);
  } else {
    e = cudaLaunchKernelEx(&cfg, fa_fwd_kernel<D, T, Q>, mq, mk, mv, p);
  }
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

template <int D, int T>
fa_status run(const void *q, const void *k, const void *v, FwdParams p,
              long long bh, cudaStream_t stream) {
  const void *kb = p.Nk > 0 ? k : q, *vb = p.Nk > 0 ? v : q;
  const int nk_map = p.Nk > 0 ? p.Nk : p.Nq;
  CUtensorMap mq, mk, mv;
  if (!encode_map<D, T>(&mq, q, p.Nq, bh) || !encode_map<D, T>(&mk, kb, nk_map, bh) ||
      !encode_map<D, T>(&mv, vb, nk_map, bh))
    return FA_ERR_CUDA;
  if constexpr (D == 64 && Elem<T>::kF8) {
    return run_shape<D, T, 1>(mq, mk, mv, p, bh, stream);
  } else {
    if constexpr (D == 64)
      if (p.Nk <= kOneTileMaxNk) return run_shape<D, T, 1>(mq, mk, mv, p, bh, stream);
    return run_shape<D, T, 2>(mq, mk, mv, p, bh, stream);
  }
}

bool aligned(const void *p, uintptr_t a);

// Streams of the host-buffer pipeline (upload, compute, download), created
// once per device.
constexpr int kPipeStreams = 3;
cudaStream_t g_pipe[kMaxDevices][kPipeStreams] = {};

fa_status pipe_streams(int dev, cudaStream_t **out) {
  std::lock_guard<std::mutex> lock(g_mutex);
  if (!g_pipe[dev][0]) {
    // published only once all three exist: a half-made set would leave null
    // (legacy default) streams in the table
    cudaStream_t made[kPipeStreams] = {};
    for (int t = 0; t < kPipeStreams; ++t)
      if (cudaStreamCreateWithFlags(&made[t], cudaStreamNonBlocking) != cudaSuccess) {
        for (int u = 0; u < t; ++u) cudaStreamDestroy(made[u]);
        return FA_ERR_CUDA;
      }
    for (int t = 0; t < kPipeStreams; ++t) g_pipe[dev][t] = made[t];
  }
  *out = g_pipe[dev];
  return FA_OK;
}

// The events of one fa_fwd_host call, destroyed when the call returns (an
// event destroyed while its record is pending is released once the record
// completes).
template <int N>
struct EventSet {
  cudaEvent_t ev[N] = {};
  int made = 0;
  bool create() {
    for (; made < N; ++made)
      if (cudaEventCreateWithFlags(&ev[made], cudaEventDisableTiming) != cudaSuccess)
        return false;
    return true;
  }
  ~EventSet() {
    for (int i = 0; i < made; ++i) cudaEventDestroy(ev[i]);
  }
};

struct WaitTestParams {
  unsigned long long timeout_ns;
  unsigned *status;
};

// One warp waits, with the kernels' bounded wait, on a phase of an mbarrier
// that expects one arrival nobody makes.
__global__ void fa_selftest_wait_kernel(const WaitTestParams p) {
  __shared__ uint64_t mbar;
  __shared__ int abort_flag;
  const uint32_t b = ptx::smem_u32(&mbar);
  if (threadIdx.x == 0) {
    ptx::mbar_init(b, 1);
    abort_flag = 0;
    ptx::fence_mbar_init();
  }
  __syncwarp();
  wait_warp(b, 0, &abort_flag, p);
}

// Encodes the maps and launches the three backward kernels: the dQ kernel
// reads Q and dO as 128-row tiles and K and V as 64-row blocks, the dK/dV
// kernel the other way round.
template <int D, int T>
fa_status run_bwd(const void *q, const void *k, const void *v, const void *dout,
                  const BwdParams &p, long long bh, cudaStream_t stream) {
  CUtensorMap mq, mk, mv, mdo, mq_b, mk_b, mv_b, mdo_b;
  if (!encode_map<D, T>(&mq, q, p.Nq, bh) || !encode_map<D, T>(&mk, k, p.Nk, bh) ||
      !encode_map<D, T>(&mv, v, p.Nk, bh) || !encode_map<D, T>(&mdo, dout, p.Nq, bh) ||
      !encode_map<D, T>(&mq_b, q, p.Nq, bh, kBwdBlk) ||
      !encode_map<D, T>(&mk_b, k, p.Nk, bh, kBwdBlk) ||
      !encode_map<D, T>(&mv_b, v, p.Nk, bh, kBwdBlk) ||
      !encode_map<D, T>(&mdo_b, dout, p.Nq, bh, kBwdBlk))
    return FA_ERR_CUDA;
  const long long rows_pad = bh * (long long)p.n_pad;
  const long long threads = rows_pad * 8;
  fa_bwd_dot_kernel<D, T><<<(unsigned)((threads + 255) / 256), 256, 0, stream>>>(p, rows_pad);
  if (cudaGetLastError() != cudaSuccess) return FA_ERR_CUDA;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kBwdThreads, 1, 1);
  cfg.stream = stream;
  cfg.gridDim = dim3((unsigned)(bh * p.n_qblk), 1, 1);
  cfg.dynamicSmemBytes = BwdQLayout<D, T>::kAlloc;
  if (cudaLaunchKernelEx(&cfg, fa_bwd_dq_kernel<D, T>, mq, mk_b, mv_b, mdo, p) != cudaSuccess)
    return FA_ERR_CUDA;
  cfg.gridDim = dim3((unsigned)(bh * p.n_kblk), 1, 1);
  cfg.dynamicSmemBytes = BwdKVLayout<D, T>::kAlloc;
  if (cudaLaunchKernelEx(&cfg, fa_bwd_dkdv_kernel<D, T>, mq_b, mk, mv, mdo_b, p) != cudaSuccess)
    return FA_ERR_CUDA;
  return FA_OK;
}

// Shared argument checks and set-up of fa_fwd_qk and fa_fwd_fp8.  Returns
// FA_OK with *launch false for an empty problem.
fa_status prepare(const void *q, const void *k, const void *v, const void *o,
                  const float *lse, int B, int H, int Nq, int Nk, int d,
                  float scale, long long *bh_out, long long *units_out,
                  int *dev_out, bool *launch) {
  *launch = false;
  if (B < 0 || H < 0 || Nq < 0 || Nk < 0) return FA_ERR_SHAPE;
  if (d != 64 && d != 128) return FA_ERR_HEADDIM;
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
  *bh_out = bh;
  *units_out = units;
  *dev_out = dev;
  *launch = true;
  return FA_OK;
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
  long long bh = 0, units = 0;
  int dev = 0;
  bool launch = false;
  fa_status st = prepare(q, k, v, o, lse, B, H, Nq, Nk, d, scale, &bh, &units,
                         &dev, &launch);
  if (st != FA_OK || !launch) return st;
  FwdParams p;
  p.o = o;
  p.lse = lse;
  p.Nq = Nq;
  p.Nk = Nk;
  p.n_units = (int)units;
  p.causal = causal ? 1 : 0;
  p.c = (float)((double)scale * 1.4426950408889634);
  p.o_scale = 1.f;
  p.timeout_ns = kTimeoutNs;
  p.status = g_status_ptr[dev];
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const bool bf16 = dtype == FA_BF16;
  if (d == 64)
    return bf16 ? run<64, kBF16>(q, k, v, p, bh, s) : run<64, kF16>(q, k, v, p, bh, s);
  return bf16 ? run<128, kBF16>(q, k, v, p, bh, s) : run<128, kF16>(q, k, v, p, bh, s);
}

fa_status fa_fwd_fp8(const void *q, const void *k, const void *v, void *o,
                     float *lse, int B, int H, int Nq, int Nk, int d, int causal,
                     float scale, float q_descale, float k_descale,
                     float v_descale, fa_stream_t stream) {
  using namespace fa;
  if (!std::isfinite(q_descale) || !std::isfinite(k_descale) ||
      !std::isfinite(v_descale) || !(q_descale > 0.f) || !(k_descale > 0.f) ||
      !(v_descale > 0.f))
    return FA_ERR_SCALE;
  long long bh = 0, units = 0;
  int dev = 0;
  bool launch = false;
  fa_status st = prepare(q, k, v, o, lse, B, H, Nq, Nk, d, scale, &bh, &units,
                         &dev, &launch);
  if (st != FA_OK || !launch) return st;
  const double c = (double)scale * (double)q_descale * (double)k_descale *
                   1.4426950408889634;
  if (!(c > 0.0) || !std::isfinite(c) || c > 3.0e38) return FA_ERR_SCALE;
  FwdParams p;
  p.o = o;
  p.lse = lse;
  p.Nq = Nq;
  p.Nk = Nk;
  p.n_units = (int)units;
  p.causal = causal ? 1 : 0;
  p.c = (float)c;
  p.o_scale = v_descale;
  p.timeout_ns = kTimeoutNs;
  p.status = g_status_ptr[dev];
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  return d == 64 ? run<64, kE4M3>(q, k, v, p, bh, s) : run<128, kE4M3>(q, k, v, p, bh, s);
}

fa_status fa_fwd_host(const void *q_h, const void *k_h, const void *v_h,
                      void *o_h, float *lse_h, void *q_d, void *k_d, void *v_d,
                      void *o_d, float *lse_d, int B, int H, int N, int d,
                      int causal, float scale, fa_dtype dtype,
                      fa_stream_t stream) {
  using namespace fa;
  if (B < 0 || H < 0 || N < 0) return FA_ERR_SHAPE;
  if (d != 64 && d != 128) return FA_ERR_HEADDIM;
  if (dtype != FA_FP16 && dtype != FA_BF16) return FA_ERR_DTYPE;
  if (!std::isfinite(scale) || !(scale > 0.f)) return FA_ERR_SCALE;
  if (B == 0 || H == 0 || N == 0) return FA_OK;
  if (!q_h || !k_h || !v_h || !o_h || !lse_h || !q_d || !k_d || !v_d || !o_d || !lse_d)
    return FA_ERR_NULL;
  if (!aligned(q_d, 16) || !aligned(k_d, 16) || !aligned(v_d, 16) || !aligned(o_d, 16) ||
      !aligned(lse_d, 4))
    return FA_ERR_ALIGN;
  const long long bh = (long long)B * (long long)H;
  if (bh > (1ll << 31) - 1) return FA_ERR_SHAPE;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_CUDA;
  fa_status st = ensure_ready(dev);
  if (st != FA_OK) return st;
  cudaStream_t *ps = nullptr;
  if ((st = pipe_streams(dev, &ps)) != FA_OK) return st;
  cudaStream_t up = ps[0], comp = ps[1], down = ps[2];
  cudaStream_t caller = reinterpret_cast<cudaStream_t>(stream);

  // chunks of whole (batch, head) problems: up to 16, each at least one
  constexpr int kMaxChunks = 16;
  const long long chunks = bh < kMaxChunks ? bh : kMaxChunks;
  const size_t row_bytes = (size_t)d * 2u;
  const size_t head_bytes = (size_t)N * row_bytes, head_lse = (size_t)N * sizeof(float);
  EventSet<2 * kMaxChunks + 2> events;
  if (!events.create()) return FA_ERR_CUDA;
  cudaEvent_t start = events.ev[0], fin = events.ev[1];
  cudaEvent_t *ev_in = events.ev + 2, *ev_out = events.ev + 2 + kMaxChunks;
  bool ok = cudaEventRecord(start, caller) == cudaSuccess &&
            cudaStreamWaitEvent(up, start, 0) == cudaSuccess &&
            cudaStreamWaitEvent(comp, start, 0) == cudaSuccess &&
            cudaStreamWaitEvent(down, start, 0) == cudaSuccess;
  // The first chunk's upload (pipeline fill) and the last chunk's kernel and
  // download (drain) are not overlapped: those two chunks take bh / 32 heads
  // each, the others split the rest evenly.
  const long long edge = chunks >= 4 ? (bh / 32 > 0 ? bh / 32 : 1) : 0;
  auto bound = [&](long long c) -> long long {   // first head of chunk c
    if (edge == 0) return bh * c / chunks;
    if (c == 0) return 0;
    if (c == chunks) return bh;
    if (c == chunks - 1) return bh - edge;
    return edge + (bh - 2 * edge) * (c - 1) / (chunks - 2);
  };
  for (long long c = 0; ok && c < chunks; ++c) {
    const long long h0 = bound(c), h1 = bound(c + 1), nh = h1 - h0;
    const size_t off = (size_t)h0 * head_bytes, bytes = (size_t)nh * head_bytes;
    const size_t loff = (size_t)h0 * head_lse, lbytes = (size_t)nh * head_lse;
    char *qd = static_cast<char *>(q_d) + off, *kd = static_cast<char *>(k_d) + off;
    char *vd = static_cast<char *>(v_d) + off, *od = static_cast<char *>(o_d) + off;
    float *ld = reinterpret_cast<float *>(reinterpret_cast<char *>(lse_d) + loff);
    ok = cudaMemcpyAsync(qd, static_cast<const char *>(q_h) + off, bytes,
                         cudaMemcpyHostToDevice, up) == cudaSuccess &&
         cudaMemcpyAsync(kd, static_cast<const char *>(k_h) + off, bytes,
                         cudaMemcpyHostToDevice, up) == cudaSuccess &&
         cudaMemcpyAsync(vd, static_cast<const char *>(v_h) + off, bytes,
                         cudaMemcpyHostToDevice, up) == cudaSuccess &&
         cudaEventRecord(ev_in[c], up) == cudaSuccess &&
         cudaStreamWaitEvent(comp, ev_in[c], 0) == cudaSuccess;
    if (!ok) break;
    st = fa_fwd_qk(qd, kd, vd, od, ld, 1, (int)nh, N, N, d, causal, scale, dtype,
                   reinterpret_cast<fa_stream_t>(comp));
    if (st != FA_OK) { ok = false; break; }
    ok = cudaEventRecord(ev_out[c], comp) == cudaSuccess &&
         cudaStreamWaitEvent(down, ev_out[c], 0) == cudaSuccess &&
         cudaMemcpyAsync(static_cast<char *>(o_h) + off, od, bytes,
                         cudaMemcpyDeviceToHost, down) == cudaSuccess &&
         cudaMemcpyAsync(reinterpret_cast<char *>(lse_h) + loff, ld, lbytes,
                         cudaMemcpyDeviceToHost, down) == cudaSuccess;
  }
  // `stream` waits for all three streams, also after a failure part way, so
  // that work the caller orders after this call never overtakes a copy this
  // call enqueued (on success the downloads come last and the other two
  // waits are already satisfied).
  for (cudaStream_t ps_t : {up, comp, down})
    if (cudaEventRecord(fin, ps_t) != cudaSuccess ||
        cudaStreamWaitEvent(caller, fin, 0) != cudaSuccess)
      ok = false;
  if (!ok) return st != FA_OK ? st : FA_ERR_CUDA;
  return FA_OK;
}

fa_status fa_fwd(const void *q, const void *k, const void *v, void *o,
                 float *lse, int B, int H, int N, int d, int causal,
                 float scale, fa_dtype dtype, fa_stream_t stream) {
  if (N < 0) return FA_ERR_SHAPE;
  return fa_fwd_qk(q, k, v, o, lse, B, H, N, N, d, causal, scale, dtype, stream);
}

size_t fa_bwd_workspace_bytes(int B, int H, int N) {
  if (B <= 0 || H <= 0 || N <= 0) return 0;
  // two fp32 arrays (LSE in exp2 units, D) of B*H heads x N rounded up to
  // whole 128-row blocks
  const size_t n_pad = ((size_t)N + fa::kBM - 1) / fa::kBM * fa::kBM;
  return 2 * (size_t)B * (size_t)H * n_pad * sizeof(float);
}

}  // extern "C"

namespace fa {
namespace {

// The host-side checks of fa_bwd that need no workspace, in the order fa_bwd
// makes them; none of them touches CUDA.  Returns FA_OK with *empty set for
// a problem with no rows.
fa_status bwd_host_checks(const void *q, const void *k, const void *v, const void *o,
                          const void *dout, const float *lse, const void *dq,
                          const void *dk, const void *dv, int B, int H, int N, int d,
                          float scale, fa_dtype dtype, bool *empty) {
  *empty = false;
  if (B < 0 || H < 0 || N < 0) return FA_ERR_SHAPE;
  if (d != 64 && d != 128) return FA_ERR_HEADDIM;
  if (dtype != FA_FP16 && dtype != FA_BF16) return FA_ERR_DTYPE;
  if (!std::isfinite(scale) || !(scale > 0.f)) return FA_ERR_SCALE;
  if (B == 0 || H == 0 || N == 0) {   // empty problem
    *empty = true;
    return FA_OK;
  }
  // B*H bounded before any product with it; N padded to whole 128-row blocks
  // must stay an int
  if ((long long)B * (long long)H > (1ll << 31) - 1) return FA_ERR_SHAPE;
  if (((long long)N + kBM - 1) / kBM * kBM > (1ll << 31) - 1) return FA_ERR_SHAPE;
  if (!q || !k || !v || !o || !lse || !dout || !dq || !dk || !dv) return FA_ERR_NULL;
  if (!aligned(dout, 16) || !aligned(dq, 16) || !aligned(dk, 16) || !aligned(dv, 16))
    return FA_ERR_ALIGN;
  return FA_OK;
}

}  // namespace
}  // namespace fa

extern "C" {

fa_status fa_bwd(const void *q, const void *k, const void *v, const void *o,
                 const void *dout, const float *lse, void *dq, void *dk, void *dv,
                 void *workspace, size_t workspace_bytes, int B, int H, int N,
                 int d, int causal, float scale, fa_dtype dtype,
                 fa_stream_t stream) {
  using namespace fa;
  // every host-side check before the first CUDA call
  bool empty = false;
  fa_status hst = bwd_host_checks(q, k, v, o, dout, lse, dq, dk, dv, B, H, N, d, scale,
                                  dtype, &empty);
  if (hst != FA_OK || empty) return hst;
  if (!workspace || !aligned(workspace, 16) ||
      workspace_bytes < fa_bwd_workspace_bytes(B, H, N))
    return FA_ERR_WORKSPACE;
  long long bh = 0, units = 0;
  int dev = 0;
  bool launch = false;
  fa_status st = prepare(q, k, v, o, lse, B, H, N, N, d, scale, &bh, &units,
                         &dev, &launch);
  if (st != FA_OK || !launch) return st;
  BwdParams p;
  p.o = o;
  p.dout = dout;
  p.lse = lse;
  p.n_pad = (int)(((long long)N + kBM - 1) / kBM * kBM);   // <= INT_MAX, checked
  p.nlse2 = static_cast<float *>(workspace);
  p.ndsum = p.nlse2 + (size_t)bh * (size_t)p.n_pad;
  p.dq = dq;
  p.dk = dk;
  p.dv = dv;
  p.Nq = N;
  p.Nk = N;
  p.n_qblk = (N + kBM - 1) / kBM;
  p.n_kblk = (N + kBN - 1) / kBN;
  p.causal = causal ? 1 : 0;
  p.c = (float)((double)scale * 1.4426950408889634);
  p.scale = scale;
  p.timeout_ns = kTimeoutNs;
  p.status = g_status_ptr[dev];
  if (bh * (long long)p.n_kblk > (1ll << 31) - 1) return FA_ERR_SHAPE;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const bool bf16 = dtype == FA_BF16;
  if (d == 64)
    return bf16 ? run_bwd<64, kBF16>(q, k, v, dout, p, bh, s)
                : run_bwd<64, kF16>(q, k, v, dout, p, bh, s);
  return bf16 ? run_bwd<128, kBF16>(q, k, v, dout, p, bh, s)
              : run_bwd<128, kF16>(q, k, v, dout, p, bh, s);
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
    case FA_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
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

fa_status fa_selftest_wait_timeout(unsigned long long timeout_ns,
                                   fa_stream_t stream) {
  using namespace fa;
  if (timeout_ns < 1000ull || timeout_ns > 1000000000ull) return FA_ERR_SHAPE;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_CUDA;
  const fa_status st = ensure_ready(dev);
  if (st != FA_OK) return st;
  WaitTestParams p;
  p.timeout_ns = timeout_ns;
  p.status = g_status_ptr[dev];
  fa_selftest_wait_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(p);
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

}  // extern "C"

namespace fa {
namespace {

// Scratch of fa_bwd_noalloc (LSE in exp2 units and D, two fp32 per padded
// query row): static device memory, one copy on every device that loads
// the library, shared by all calls.
constexpr long long kNoAllocMaxRows = FA_BWD_NOALLOC_MAX_ROWS;
static __device__ __align__(256) float g_noalloc_dsum[2 * kNoAllocMaxRows];

std::mutex g_noalloc_mutex;
void *g_noalloc_ptr[kMaxDevices] = {};

// The array's device address for device `dev` (current), looked up once.
fa_status noalloc_scratch(int dev, void **out) {
  if (dev < 0 || dev >= kMaxDevices) return FA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  if (!g_noalloc_ptr[dev]) {
    void *ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_dsum) != cudaSuccess || !ptr)
      return FA_ERR_CUDA;
    g_noalloc_ptr[dev] = ptr;
  }
  *out = g_noalloc_ptr[dev];
  return FA_OK;
}

}  // namespace
}  // namespace fa

extern "C" {

fa_status fa_bwd_noalloc(const void *q, const void *k, const void *v,
                         const void *o, const void *dout, const float *lse,
                         void *dq, void *dk, void *dv, int B, int H, int N,
                         int d, int causal, float scale, fa_dtype dtype,
                         fa_stream_t stream) {
  using namespace fa;
  // fa_bwd's host-side checks first, so that a bad argument gets fa_bwd's
  // error and nothing touches CUDA before they pass
  bool empty = false;
  const fa_status hst = bwd_host_checks(q, k, v, o, dout, lse, dq, dk, dv, B, H, N, d,
                                        scale, dtype, &empty);
  if (hst != FA_OK || empty) return hst;
  // B*H < 2^31 and n_pad < 2^31 (checked above): the product fits in 64 bits
  const long long n_pad = ((long long)N + kBM - 1) / kBM * kBM;
  if ((long long)B * (long long)H * n_pad > kNoAllocMaxRows) return FA_ERR_WORKSPACE;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_CUDA;
  void *scratch = nullptr;
  const fa_status st = noalloc_scratch(dev, &scratch);
  if (st != FA_OK) return st;
  return fa_bwd(q, k, v, o, dout, lse, dq, dk, dv, scratch,
                2 * (size_t)kNoAllocMaxRows * sizeof(float), B, H, N, d, causal,
                scale, dtype, stream);
}

}  // extern "C"
