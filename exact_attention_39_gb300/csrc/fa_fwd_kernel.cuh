// fa_fwd_kernel.cuh -- the attention forward kernel for sm_103a.
//
// What it computes: O = softmax(scale * Q K^T [+ causal mask]) V and the
// per-row logsumexp, for one (batch, head) problem per group of CTAs.  The
// pages describe the method as splitting the computation into blocks that
// fit in on-chip memory so the attention matrix never goes to HBM
// (zzycbzc.com/news/393333, section "FlashAttention的技术革命"; the
// "0 MB (recompute)" column of the benchmarks page's Flash Attention 2
// memory table).  Keeping only a running row maximum and a running row sum
// (the online softmax) is what makes one pass over the key blocks exact.
//
// Shape of one CTA (a "work unit" = 256 query rows of one head):
//   warps 0-3  softmax warpgroup for query tile 0 (rows q0 .. q0+127)
//   warps 4-7  softmax warpgroup for query tile 1 (rows q0+128 .. q0+255)
//              thread t of a warpgroup owns query row t = TMEM lane t
//   warp  8    TMA producer: Q tiles once, then K/V blocks into a ring
//   warp  9    TMEM allocator and tcgen05 MMA issuer (one thread)
//   warps 10-11 idle (they complete the third warpgroup, which lets the
//              register budget be moved to the softmax warpgroups)
//
// Per key block j the MMA thread issues, for D = 64 (P has TMEM columns of
// its own):
//   S_0 = Q_0 K_{j+1}^T, S_1 = Q_1 K_{j+1}^T   once both warpgroups have read
//                                               their block-j scores;
//   O_0 += P_0 V_j,      O_1 += P_1 V_j        once both have written P(j);
// so the next scores are computed while softmax works on the current ones.
// For D = 128 (P over the first columns of S_i) it issues, tile by tile,
// O_i += P_i V_j and then S_i = Q_i K_{j+1}^T: the tensor pipe runs one
// thread's MMAs in order, so the product reads P_i before the next scores
// overwrite it.  A commit after each O_i += P_i V_j (o_done) tells softmax
// warpgroup i that it may rescale O_i and overwrite P_i.
//
// TMEM (512 columns, fp32 cells, 128 lanes):
//   S_i  at columns i*128 .. i*128+127   (scores of tile i, one row per lane)
//   O_i  at columns 256 + i*D           (output accumulator of tile i)
//   P_i  (16-bit probabilities, two per cell) at 384 + i*64 for D = 64; for
//        D = 128 the accumulators fill TMEM and P_i overwrites the first 64
//        columns of S_i, which its own thread has finished reading.
//
// Shared memory: two Q tiles, then a ring of K and V blocks; every tile is
// stored as 128-row x 64-element (128-byte) chunks in the TMA 128-byte
// swizzle, which is also the layout the MMA's matrix descriptors name.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <math_constants.h>

#include "ptx.cuh"

namespace fa {

constexpr int kBM = 128;                 // query rows per tile
constexpr int kBN = 128;                 // keys per block
constexpr int kTmemCols = 512;           // TMEM columns of an SM

// Shape of a CTA with Q query tiles (Q softmax warpgroups and one control
// warpgroup).  Q = 2 is the default: one CTA per SM.  Q = 1 (D = 64: 16-bit
// inputs with at most 4096 keys, and every e4m3 launch) halves shared memory
// and TMEM so that two CTAs share an SM and one CTA's set-up, first loads,
// epilogue and exit overlap the other's key blocks.
template <int Q>
struct CtaShape {
  static constexpr int kThreads = 128 * Q + 128;
  static constexpr int kLoadWarp = 4 * Q;
  static constexpr int kMmaWarp = 4 * Q + 1;   // the warpgroup's last two warps idle
  static constexpr int kMinBlocks = Q == 1 ? 2 : 1;
  // Register split (setmaxnreg): the control warpgroup gives registers to
  // the softmax warpgroups within the launch's budget, 65536 / kMinBlocks
  // per CTA: Q = 2: 128*88 + 256*208 = 64512 <= 384*168; Q = 1:
  // 128*56 + 128*200 = 32768 = 256*128.
  static constexpr uint32_t kRegsControl = Q == 2 ? 88 : 56;
  static constexpr uint32_t kRegsSoftmax = Q == 2 ? 208 : 200;
  static_assert(Q == 1 || Q == 2, "one or two query tiles per CTA");
  static_assert(128 * kRegsControl + 128 * Q * kRegsSoftmax <=
                (uint32_t)(65536 / kMinBlocks / kThreads) / 8u * 8u * kThreads,
                "register split exceeds the launch budget");
};
// Compatibility names for the default shape.
constexpr int kNumQ = 2;
constexpr int kRowsPerCta = kBM * kNumQ;
// A rescale of O is skipped while the running maximum grows by at most this
// much (log2 units): probabilities then stay below 2^8, which fp16, bf16 and
// the fp32 accumulators hold exactly as well as values below 1.
constexpr float kRescaleThreshold = 8.0f;
// Causal work order: a group of heads holds at most this many bytes of K and
// V (so that they stay in the 129 MB L2 beside Q and O) and at most
// kCausalMaxHeadGroup heads.
constexpr long long kCausalGroupKVBytes = 64ll << 20;
constexpr int kCausalMaxHeadGroup = 32;

enum : unsigned { kStatusTimeout = 1u };

struct FwdParams {
  void *o;            // [BH, Nq, D] output
  float *lse;         // [BH, Nq] output
  int Nq, Nk;         // query and key rows per head
  int n_units;        // work units per head: ceil(Nq / 256)
  int head_group;     // causal work order: heads per group (see fa_fwd_kernel)
  int causal;
  float c;            // scale * log2(e) (* q and k descales for e4m3), > 0
  float o_scale;      // multiplies O before the division by l (v descale)
  unsigned long long timeout_ns;
  unsigned *status;   // device status word (timeout flags)
};

// Element types of Q, K, V and of P in the second product.
enum ElemType : int { kF16 = 0, kBF16 = 1, kE4M3 = 2 };

template <int T> struct Elem;
template <> struct Elem<kF16> {
  static constexpr int kBytes = 2;
  static constexpr int kMmaK = 16;          // K of one tcgen05.mma (32 bytes)
  static constexpr uint32_t kFmt = 0;       // instruction-descriptor format
  static constexpr bool kF8 = false;
};
template <> struct Elem<kBF16> {
  static constexpr int kBytes = 2;
  static constexpr int kMmaK = 16;
  static constexpr uint32_t kFmt = 1;
  static constexpr bool kF8 = false;
};
template <> struct Elem<kE4M3> {
  static constexpr int kBytes = 1;
  static constexpr int kMmaK = 32;
  static constexpr uint32_t kFmt = 0;
  static constexpr bool kF8 = true;
};

template <int D, int T, int Q = 2>
struct Layout {
  using E = Elem<T>;
  // Tiles are stored as chunks of kBM rows x kSwz bytes in the TMA swizzle of
  // the same width (128 bytes; 64 when a whole row is only 64 bytes).
  static constexpr int kRowBytes = D * E::kBytes;
  static constexpr int kSwz = kRowBytes < 128 ? kRowBytes : 128;
  static constexpr int kChunkElems = kSwz / E::kBytes;
  static constexpr int kChunks = D / kChunkElems;
  static constexpr int kChunkBytes = kBM * kSwz;
  static constexpr int kTileBytes = kChunks * kChunkBytes;
  static constexpr int kSBO = 8 * kSwz;                 // 8-row swizzle atom
  static constexpr uint64_t kSwzMode = kSwz == 128 ? 2 : 4;   // descriptor code
  // Q = 1 keeps two stages so that two CTAs fit the SM's shared memory
  static constexpr int kStages = Q == 1 ? 2 : (kTileBytes <= 16384 ? 4 : 2);
  static constexpr int kQ = 0;
  static constexpr int kK = kQ + Q * kTileBytes;
  static constexpr int kV = kK + kStages * kTileBytes;
  static constexpr int kBars = kV + kStages * kTileBytes;
  // barrier indices
  static constexpr int bQFull = 0;
  static constexpr int bKFull = 1;
  static constexpr int bVFull = bKFull + kStages;
  static constexpr int bKVEmpty = bVFull + kStages;  // K and V (K alone when split)
  // One query tile: K and V of a stage land and free on barriers of their
  // own, so that K_{j+2} is loaded as soon as the scores of block j are done
  // instead of after O += P V_j (with two stages the ring could not refill
  // within one block; the next scores waited for their K).
  static constexpr bool kSplitKV = Q == 1;
  static constexpr int bVEmpty = bKVEmpty + kStages;  // V (split only)
  static constexpr int bSFull = bVEmpty + (kSplitKV ? kStages : 0);   // S_i ready (MMA commit)
  static constexpr int bSFree = bSFull + Q;          // S_i read into registers
  static constexpr int bPFull = bSFree + Q;           // P_i written, O_i rescaled
  static constexpr int bODone = bPFull + Q;           // O_i += P_i V_j done (commit)
  static constexpr int bDrain = bODone + Q;
  static constexpr int kNumBars = bDrain + 1;
  static constexpr int kMisc = kBars + kNumBars * 8;   // tmem base, abort flag
  static constexpr int kBytes = kMisc + 16;
  static constexpr int kAlloc = kBytes + 1024;         // room to align to 1 KB
  // TMEM columns of one tile's P (four 8-bit or two 16-bit values a cell).
  static constexpr int kPCols = kBN * E::kBytes / 4;
  // When P fits beside the accumulators it has TMEM columns of its own, so
  // the MMA for the next block's scores may overwrite S_i as soon as softmax
  // has read it.
  // TMEM columns the CTA allocates (a power of two, at least 32)
  static constexpr int kTmem = Q == 2 ? kTmemCols : kTmemCols / 2;
  static constexpr bool kEarlyS = Q * (kBN + D + kPCols) <= kTmem;
  // With the early scores the MMA thread keeps its per-block waits to three:
  // K and V of a stage land on one barrier, and one barrier each counts both
  // warpgroups' "scores read" and "P written" arrivals.  (The thread shares
  // its sub-partition with two softmax warps, so each wait it makes costs
  // issue slots that delay every later MMA.)
  static constexpr bool kMerged = kEarlyS;
  // TMEM columns: S_i, then O_i, then (early scores) P_i
  __host__ __device__ static constexpr uint32_t tS(int i) { return i * kBN; }
  __host__ __device__ static constexpr uint32_t tO(int i) { return Q * kBN + i * D; }
  __host__ __device__ static constexpr uint32_t tP(int i) {
    return kEarlyS ? Q * (kBN + D) + i * kPCols : i * kBN;
  }
};

// Instruction descriptor of tcgen05.mma (kind::f16 or kind::f8f6f4): fp32
// accumulator, A and B of one format (f16 0 / bf16 1, or e4m3 0), A K-major,
// B K-major or MN-major, M x N.
__host__ __device__ constexpr uint32_t make_idesc(int M, int N, uint32_t fmt,
                                                  bool b_mn_major) {
  return (1u << 4)                                  // D format: f32
         | (fmt << 7)                               // A format
         | (fmt << 10)                              // B format
         | ((b_mn_major ? 1u : 0u) << 16)           // B major-ness
         | ((uint32_t)(N >> 3) << 17)               // N / 8
         | ((uint32_t)(M >> 4) << 24);              // M / 16
}

// Shared-memory matrix descriptor: start address, leading- and stride-
// dimension byte offsets, the fixed version field, and the swizzle mode
// (2: 128-byte swizzle, 4: 64-byte swizzle).
__device__ __forceinline__ uint64_t make_sdesc(uint32_t saddr, uint32_t lbo,
                                               uint32_t sbo, uint64_t mode) {
  uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;
  d |= mode << 61;
  return d;
}

// A bounded wait on an mbarrier phase.  Gives up when the CTA's abort flag is
// set or after timeout_ns of global time; on a timeout it sets the abort flag
// and records the timeout in the device status word.  (P: any parameter
// block with timeout_ns and status.)
template <class P>
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity,
                                           volatile int *abort_flag,
                                           const P &p) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = ptx::globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    if ((it & 31u) == 0) {
      if (*abort_flag) return false;
      if (ptx::globaltimer_ns() - t0 > p.timeout_ns) {
        *abort_flag = 1;
        atomicOr(p.status, (unsigned)kStatusTimeout);
        return false;
      }
    }
  }
}

// wait_phase executed by all 32 lanes of a warp, with one warp-wide result.
template <class P>
__device__ __forceinline__ bool wait_warp(uint32_t bar, uint32_t parity,
                                          volatile int *abort_flag,
                                          const P &p) {
  const bool ok = wait_phase(bar, parity, abort_flag, p);
  return __all_sync(0xffffffffu, ok);
}

// A wait used only while draining on the way out: bounded by the timeout
// alone (it must not give up just because the CTA is aborting).
template <class P>
__device__ __forceinline__ bool wait_drain(uint32_t bar, uint32_t parity,
                                           const P &p) {
  const uint64_t t0 = ptx::globaltimer_ns();
  for (;;) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    if (ptx::globaltimer_ns() - t0 > p.timeout_ns) {
      atomicOr(p.status, (unsigned)kStatusTimeout);
      return false;
    }
  }
}

// kSkip (causal launches of the two-tile shape with merged barriers): a
// tile that sees no key of the CTA's last block -- it lies wholly past the
// tile's diagonal -- gets neither scores nor products for it.  A separate
// instantiation, so that the others keep exactly their code.
template <int D, int T, int Q, bool kSkip = false>
__global__ void __launch_bounds__(CtaShape<Q>::kThreads, CtaShape<Q>::kMinBlocks)
    fa_fwd_kernel(const __grid_constant__ CUtensorMap tmQ,
                  const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV,
                  const FwdParams p) {
  using L = Layout<D, T, Q>;
  using C = CtaShape<Q>;
  constexpr int kNumQ = Q;
  constexpr int kRowsPerCta = Q * kBM;
  constexpr int kLoadWarp = C::kLoadWarp;
  constexpr int kMmaWarp = C::kMmaWarp;
  using E = Elem<T>;
  constexpr bool kF8 = E::kF8;
  constexpr bool kOutBF16 = T != kF16;   // e4m3 inputs give a bf16 output
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw = ptx::smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t *smem = smem_raw + (sbase - raw);
  const uint32_t bars = sbase + L::kBars;
  auto bar = [&](int idx) -> uint32_t { return bars + 8u * (uint32_t)idx; };
  volatile uint32_t *tmem_slot = reinterpret_cast<volatile uint32_t *>(smem + L::kMisc);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::kMisc + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // ---- work unit: (head bh, unit of Q * 128 query rows).  Non-causal: the
  // units of a head are consecutive, so the CTAs resident at one time share
  // K/V blocks in L2.  Causal: units differ in length, so the grid runs, in
  // groups of p.head_group heads, the longest unit of every head of the
  // group first, then the next longest, and so on (longest-processing-time
  // order keeps the tail short; the host sizes a group so that its K and V
  // stay in L2 while it runs).
  int bh, unit;
  if (p.causal) {
    const int nbh = (int)(gridDim.x / (unsigned)p.n_units);
    const int G = p.head_group;
    const int per_group = G * p.n_units;
    const int g = (int)blockIdx.x / per_group, r = (int)blockIdx.x % per_group;
    const int heads = min(G, nbh - g * G);
    bh = g * G + r % heads;
    unit = p.n_units - 1 - r / heads;
  } else {
    bh = (int)(blockIdx.x / (unsigned)p.n_units);
    unit = (int)(blockIdx.x % (unsigned)p.n_units);
  }
  const int q0 = unit * kRowsPerCta;
  int kv_end = p.Nk;
  if (p.causal) kv_end = min(p.Nk, q0 + kRowsPerCta + (p.Nk - p.Nq));
  const int nb = kv_end > 0 ? (kv_end + kBN - 1) / kBN : 0;
  // Key blocks of query tile i (kSkip): those up to the block that holds its
  // last row's diagonal (the last tile's are nb).
  auto tile_blocks = [&](int i) -> int {
    const int end = min(p.Nk, q0 + (i + 1) * kBM + (p.Nk - p.Nq));
    return end > 0 ? (end + kBN - 1) / kBN : 0;
  };
  static_assert(!kSkip || (Layout<D, T, Q>::kMerged && Q == 2), "skip: merged two-tile shape");
  // The non-causal two-tile kernels for 16-bit inputs announce "scores read"
  // and "P written" with one arrival per softmax warp, after a warp barrier,
  // instead of one per thread (measured on the GB300: +0.6 % at B8 H32 N8192
  // d64, +0.1 % at d = 128; the causal and e4m3 kernels lost 5 and 10 % with
  // it and keep per-thread arrivals).
  constexpr bool kWarpArrive = Q == 2 && !kSkip && !kF8;

  // ---- set-up: TMEM, barriers
  if (warp == kMmaWarp) {
    ptx::tmem_alloc(sbase + L::kMisc, L::kTmem);
    ptx::tmem_relinquish();
  }
  if (threadIdx.x == 0) {
    ptx::mbar_init(bar(L::bQFull), 1);
    for (int s = 0; s < L::kStages; ++s) {
      ptx::mbar_init(bar(L::bKFull + s), 1);   // K, or K and V when merged
      ptx::mbar_init(bar(L::bVFull + s), 1);
      ptx::mbar_init(bar(L::bKVEmpty + s), 1);
      if (L::kSplitKV) ptx::mbar_init(bar(L::bVEmpty + s), 1);
    }
    for (int i = 0; i < kNumQ; ++i) {
      ptx::mbar_init(bar(L::bSFull + i), 1);
      // merged: barrier 0 of each pair counts both warpgroups
      // arrivals per tile: one per softmax warp (kWarpArrive) or per thread
      constexpr int kArr = kWarpArrive ? 4 : kBM;
      ptx::mbar_init(bar(L::bSFree + i), L::kMerged ? kNumQ * kArr : kArr);
      ptx::mbar_init(bar(L::bPFull + i), L::kMerged ? kNumQ * kArr : kArr);
      ptx::mbar_init(bar(L::bODone + i), 1);
    }
    ptx::mbar_init(bar(L::bDrain), 1);
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == kLoadWarp && lane == 0) {
    ptx::prefetch_tmap(&tmQ);
    ptx::prefetch_tmap(&tmK);
    ptx::prefetch_tmap(&tmV);
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp >= 4 * Q) {
   ptx::regs_dec<C::kRegsControl>();
   // The producer and MMA warps run their loops with all 32 lanes, so every
   // operand is warp-uniform; one elected lane issues each copy, MMA and
   // commit (a commit tracks the MMAs of the lane that issues it).
   if (warp == kLoadWarp) {
    // ================================================= TMA producer
    if (nb > 0) {
      const bool leader = ptx::elect_one();
      const uint64_t pol_q = ptx::policy_evict_first();
      const uint64_t pol_kv = ptx::policy_evict_last();
      if (leader) {
        ptx::mbar_arrive_expect_tx(bar(L::bQFull), kNumQ * L::kTileBytes);
        for (int i = 0; i < kNumQ; ++i)
          for (int c = 0; c < L::kChunks; ++c)
            ptx::tma_load_3d(sbase + L::kQ + i * L::kTileBytes + c * L::kChunkBytes,
                             &tmQ, bar(L::bQFull), c * L::kChunkElems, q0 + i * kBM, bh, pol_q);
      }
      if constexpr (L::kSplitKV) {
        // K_{j+1} ahead of V_j: a K stage frees when its scores are done, a
        // V stage when its product is.
        auto load = [&](int j, bool is_v) -> bool {
          const int st = j % L::kStages;
          const int use = j / L::kStages;
          const int empty = is_v ? L::bVEmpty : L::bKVEmpty;
          const int full = is_v ? L::bVFull : L::bKFull;
          if (use > 0 && !wait_warp(bar(empty + st), (use - 1) & 1, abort_flag, p))
            return false;
          if (leader) {
            ptx::mbar_arrive_expect_tx(bar(full + st), L::kTileBytes);
            for (int c = 0; c < L::kChunks; ++c)
              ptx::tma_load_3d(sbase + (is_v ? L::kV : L::kK) + st * L::kTileBytes +
                                   c * L::kChunkBytes,
                               is_v ? &tmV : &tmK, bar(full + st), c * L::kChunkElems,
                               j * kBN, bh, pol_kv);
          }
          return true;
        };
        int k_issued = 0, v_issued = 0;
        if (load(0, false)) {
          k_issued = 1;
          for (int j = 0; j < nb; ++j) {
            if (j + 1 < nb) {
              if (!load(j + 1, false)) break;
              k_issued = j + 2;
            }
            if (!load(j, true)) break;
            v_issued = j + 1;
          }
        }
        wait_drain(bar(L::bQFull), 0, p);
        for (int j = max(k_issued - L::kStages, 0); j < k_issued; ++j)
          wait_drain(bar(L::bKFull + j % L::kStages), (uint32_t)(j / L::kStages) & 1u, p);
        for (int j = max(v_issued - L::kStages, 0); j < v_issued; ++j)
          wait_drain(bar(L::bVFull + j % L::kStages), (uint32_t)(j / L::kStages) & 1u, p);
      } else {
      int issued = 0;
      for (int j = 0; j < nb; ++j) {
        const int st = j % L::kStages;
        const int use = j / L::kStages;
        if (use > 0 &&
            !wait_warp(bar(L::bKVEmpty + st), (use - 1) & 1, abort_flag, p))
          break;
        if (leader) {
          const uint32_t vbar = bar(L::kMerged ? L::bKFull + st : L::bVFull + st);
          ptx::mbar_arrive_expect_tx(bar(L::bKFull + st),
                                     L::kMerged ? 2 * L::kTileBytes : L::kTileBytes);
          for (int c = 0; c < L::kChunks; ++c)
            ptx::tma_load_3d(sbase + L::kK + st * L::kTileBytes + c * L::kChunkBytes,
                             &tmK, bar(L::bKFull + st), c * L::kChunkElems, j * kBN, bh, pol_kv);
          if (!L::kMerged) ptx::mbar_arrive_expect_tx(vbar, L::kTileBytes);
          for (int c = 0; c < L::kChunks; ++c)
            ptx::tma_load_3d(sbase + L::kV + st * L::kTileBytes + c * L::kChunkBytes,
                             &tmV, vbar, c * L::kChunkElems, j * kBN, bh, pol_kv);
        }
        issued = j + 1;
      }
      // Drain: every copy issued has landed before the CTA may exit
      // (returns at once on the normal path).
      wait_drain(bar(L::bQFull), 0, p);
      for (int j = issued - L::kStages; j < issued; ++j) {
        if (j < 0) continue;
        const int st = j % L::kStages;
        const uint32_t ph = (uint32_t)(j / L::kStages) & 1u;
        wait_drain(bar(L::bKFull + st), ph, p);
        if (!L::kMerged) wait_drain(bar(L::bVFull + st), ph, p);
      }
      }
    }
  } else if (warp == kMmaWarp) {
    // ================================================= MMA issuer
    if (nb > 0) {
      const bool leader = ptx::elect_one();
      constexpr uint32_t idesc_s = make_idesc(kBM, kBN, E::kFmt, false);
      constexpr uint32_t idesc_o = make_idesc(kBM, D, E::kFmt, true);
      // Descriptors are built once; stepping through a tile only adds to the
      // 14-bit start-address field (address >> 4, all smem offsets < 256 KB).
      const uint64_t dq0 = make_sdesc(sbase + L::kQ, 16, L::kSBO, L::kSwzMode);
      const uint64_t dk0 = make_sdesc(sbase + L::kK, 16, L::kSBO, L::kSwzMode);
      const uint64_t dv0 = make_sdesc(sbase + L::kV, L::kChunkBytes, L::kSBO, L::kSwzMode);
      // S_i = Q_i K_st^T, then a commit on s_full[i]
      auto issue_s = [&](int i, int st) {
        const uint64_t dq = dq0 + (uint64_t)((i * L::kTileBytes) >> 4);
        const uint64_t dk = dk0 + (uint64_t)((st * L::kTileBytes) >> 4);
        if (leader) {
#pragma unroll
          for (int kk = 0; kk < D / E::kMmaK; ++kk) {
            // one MMA step covers 32 bytes of K: inside a swizzle row the
            // start address moves by 32 bytes, across chunks by a chunk
            constexpr int kStepsPerChunk = L::kSwz / 32;
            const uint32_t off = ((kk / kStepsPerChunk) * L::kChunkBytes +
                                  (kk % kStepsPerChunk) * 32) >> 4;
            if constexpr (kF8)
              ptx::mma_ss_f8(tmem + L::tS(i), dq + off, dk + off, idesc_s, kk > 0);
            else
              ptx::mma_ss(tmem + L::tS(i), dq + off, dk + off, idesc_s, kk > 0);
          }
          ptx::mma_commit(bar(L::bSFull + i));
        }
      };
      // O_i (+)= P_i V_st, then a commit on o_done[i]
      auto issue_pv = [&](int i, int st, bool acc) {
        const uint64_t dv = dv0 + (uint64_t)((st * L::kTileBytes) >> 4);
        if (leader) {
#pragma unroll
          for (int kk = 0; kk < kBN / E::kMmaK; ++kk) {
            // K step of kMmaK keys: 8 TMEM columns of P, kMmaK swizzle rows of V
            const uint64_t dvk = dv + (uint64_t)((kk * E::kMmaK * L::kSwz) >> 4);
            if constexpr (kF8)
              ptx::mma_ts_f8(tmem + L::tO(i), tmem + L::tP(i) + kk * 8, dvk, idesc_o,
                             (acc || kk > 0) ? 1u : 0u);
            else
              ptx::mma_ts(tmem + L::tO(i), tmem + L::tP(i) + kk * 8, dvk, idesc_o,
                          (acc || kk > 0) ? 1u : 0u);
          }
          ptx::mma_commit(bar(L::bODone + i));
        }
      };
      bool ok = wait_warp(bar(L::bQFull), 0, abort_flag, p) &&
                wait_warp(bar(L::bKFull + 0), 0, abort_flag, p);
      if constexpr (kSkip) {
        // tile 0 sees blocks 0 .. nb0-1, tile 1 all nb
        const int nb0 = tile_blocks(0);
        if (ok) {
          ptx::tc_fence_after();
          if (nb0 > 0) issue_s(0, 0);
          issue_s(1, 0);
        }
        for (int j = 0; ok && j < nb; ++j) {
          const int st = j % L::kStages;
          const int st2 = (j + 1) % L::kStages;
          if (j + 1 < nb) {
            if (!wait_warp(bar(L::bKFull + st2), ((j + 1) / L::kStages) & 1, abort_flag, p) ||
                !wait_warp(bar(L::bSFree), j & 1, abort_flag, p))
              break;
            ptx::tc_fence_after();
            if (j + 1 < nb0) issue_s(0, st2);
            issue_s(1, st2);
          }
          // both warpgroups have written P(j), or (tile 0 past its diagonal)
          // arrived without one
          if (!wait_warp(bar(L::bPFull), j & 1, abort_flag, p)) break;
          ptx::tc_fence_after();
          if (j < nb0) issue_pv(0, st, j > 0);
          issue_pv(1, st, j > 0);
          if (leader) ptx::mma_commit(bar(L::bKVEmpty + st));
        }
      } else {
      if (ok) {
        ptx::tc_fence_after();
        for (int i = 0; i < kNumQ; ++i) issue_s(i, 0);
        if (L::kSplitKV && leader) ptx::mma_commit(bar(L::bKVEmpty + 0));
      }
      if constexpr (L::kMerged) {
        for (int j = 0; ok && j < nb; ++j) {
          const int st = j % L::kStages;
          const int st2 = (j + 1) % L::kStages;
          if (j + 1 < nb) {
            // Scores of block j+1 once K_{j+1} has landed and both warpgroups
            // have their block-j scores in registers.
            if (!wait_warp(bar(L::bKFull + st2), ((j + 1) / L::kStages) & 1, abort_flag, p) ||
                !wait_warp(bar(L::bSFree), j & 1, abort_flag, p))
              break;
            ptx::tc_fence_after();
            for (int i = 0; i < kNumQ; ++i) issue_s(i, st2);
            if (L::kSplitKV && leader) ptx::mma_commit(bar(L::bKVEmpty + st2));
          }
          // both warpgroups have written P(j); V_j landed (with K_j unless split)
          if (!wait_warp(bar(L::bPFull), j & 1, abort_flag, p)) break;
          if (L::kSplitKV &&
              !wait_warp(bar(L::bVFull + st), (j / L::kStages) & 1, abort_flag, p))
            break;
          ptx::tc_fence_after();
          for (int i = 0; i < kNumQ; ++i) issue_pv(i, st, j > 0);
          if (leader) ptx::mma_commit(bar(L::kSplitKV ? L::bVEmpty + st : L::bKVEmpty + st));
        }
      } else {
        for (int j = 0; ok && j < nb; ++j) {
          const int st = j % L::kStages;
          const int st2 = (j + 1) % L::kStages;
          const bool more = j + 1 < nb;
          if (L::kEarlyS && more) {
            // Scores of block j+1 as soon as each softmax warpgroup has its
            // block-j scores in registers.
            if (!wait_warp(bar(L::bKFull + st2), ((j + 1) / L::kStages) & 1, abort_flag, p)) break;
            for (int i = 0; i < kNumQ && ok; ++i) {
              if (!wait_warp(bar(L::bSFree + i), j & 1, abort_flag, p)) { ok = false; break; }
              ptx::tc_fence_after();
              issue_s(i, st2);
            }
            if (!ok) break;
          }
          if (!wait_warp(bar(L::bVFull + st), (j / L::kStages) & 1, abort_flag, p)) break;
          for (int i = 0; i < kNumQ; ++i) {
            if (!wait_warp(bar(L::bPFull + i), j & 1, abort_flag, p)) { ok = false; break; }
            ptx::tc_fence_after();
            issue_pv(i, st, j > 0);
            if (i == kNumQ - 1 && leader) ptx::mma_commit(bar(L::bKVEmpty + st));
            if (!L::kEarlyS && more) {
              // P_i shares columns with S_i: the next scores go in only after
              // O_i += P_i V_j (the tensor pipe runs one thread's MMAs in order).
              if (i == 0) {
                if (!wait_warp(bar(L::bKFull + st2), ((j + 1) / L::kStages) & 1,
                               abort_flag, p)) { ok = false; break; }
                ptx::tc_fence_after();
              }
              issue_s(i, st2);
            }
          }
        }
      }
      }
      // Every MMA issued has completed before TMEM is released.
      if (leader) ptx::mma_commit(bar(L::bDrain));
      wait_drain(bar(L::bDrain), 0, p);
    }
   }
  } else {
    // ================================================= softmax warpgroups
    ptx::regs_inc<C::kRegsSoftmax>();
    // The two-tile kernels for 16-bit inputs at D = 64 load S and store P
    // 64 columns an instruction (measured on the GB300: +1.5 to +2.4 %
    // non-causal and +1.0 to +1.2 % causal at N = 2048..8192); the e4m3 and
    // D = 128 instantiations keep 32-column loads and stores, which measured
    // faster for them (e4m3 -1 % with the wide forms).
    constexpr bool kWideLdSt = D == 64 && !kF8 && Q == 2 && L::kPCols == 64;
    const int i = warp >> 2;                  // query tile of this warpgroup
    const int r = threadIdx.x & 127;          // row within the tile = TMEM lane
    const int row = q0 + i * kBM + r;         // query row within the head
    const uint32_t lane_off = (uint32_t)(32 * (warp & 3)) << 16;
    const uint32_t tS = tmem + lane_off + L::tS(i);
    const uint32_t tO = tmem + lane_off + L::tO(i);
    const uint32_t tP = tmem + lane_off + L::tP(i);
    const float c = p.c;
    // keys [0, key_lim) are visible to this row
    const int key_lim = p.causal ? min(p.Nk, row + 1 + (p.Nk - p.Nq)) : p.Nk;
    float m = -CUDART_INF_F;   // running max of the scaled logits (log2 units)
    float l = 0.f;             // running sum of exp2(logit - m)
    bool ok = true;

    const float2 c2 = make_float2(c, c);
    // blocks this tile sees (kSkip: tile 0 may see one fewer than the CTA)
    int nb_i = nb;
    if constexpr (kSkip) nb_i = tile_blocks(i);
    for (int j = 0; j < nb_i; ++j) {
      if (!wait_phase(bar(L::bSFull + i), j & 1, abort_flag, p)) { ok = false; break; }
      ptx::tc_fence_after();
      uint32_t s[kBN];
      if constexpr (kWideLdSt) {
#pragma unroll
        for (int cc = 0; cc < kBN / 64; ++cc) ptx::tmem_ld64(tS + cc * 64, &s[cc * 64]);
        ptx::tmem_wait_ld();
#pragma unroll
        for (int cc = 0; cc < kBN / 64; ++cc) ptx::reg_fence64(&s[cc * 64]);
      } else {
#pragma unroll
        for (int cc = 0; cc < kBN / 32; ++cc)
          ptx::tmem_ld32(tS + cc * 32, *reinterpret_cast<uint32_t(*)[32]>(&s[cc * 32]));
        ptx::tmem_wait_ld();
#pragma unroll
        for (int cc = 0; cc < kBN / 32; ++cc)
          ptx::reg_fence32(*reinterpret_cast<uint32_t(*)[32]>(&s[cc * 32]));
      }
      if (L::kEarlyS) {
        ptx::tc_fence_before();
        if constexpr (kWarpArrive) {
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive(bar(L::bSFree + (L::kMerged ? 0 : i)));
        } else {
          ptx::mbar_arrive(bar(L::bSFree + (L::kMerged ? 0 : i)));
        }
      }
      float *sf = reinterpret_cast<float *>(s);

      const int lim = key_lim - j * kBN;   // columns >= lim are masked
      if (lim < kBN) {
#pragma unroll
        for (int cc = 0; cc < kBN; ++cc)
          if (cc >= lim) sf[cc] = -CUDART_INF_F;
      }
      // row maximum: eight independent chains of three-input max
      float mx[8];
#pragma unroll
      for (int t = 0; t < 8; ++t) mx[t] = sf[t];
#pragma unroll
      for (int cc = 8; cc < kBN; cc += 16) {
#pragma unroll
        for (int t = 0; t < 8; ++t)
          mx[t] = ptx::fmax3(mx[t], sf[cc + t], cc + 8 + t < kBN ? sf[cc + 8 + t] : sf[t]);
      }
      const float m_blk = ptx::fmax3(ptx::fmax3(mx[0], mx[1], mx[2]),
                                     ptx::fmax3(mx[3], mx[4], mx[5]),
                                     fmaxf(mx[6], mx[7])) * c;
      const float m_new = fmaxf(m, m_blk);
      float m_use, alpha;
      if (m_new == -CUDART_INF_F) {        // nothing visible yet
        m_use = 0.f;
        alpha = 1.f;
      } else if (m_new - m > kRescaleThreshold) {
        m_use = m_new;
        alpha = ptx::ex2_approx(m - m_new);   // 0 when m is -inf
      } else {
        m_use = m;
        alpha = 1.f;
      }
      // p = 2^(s*c - m): scale and shift two at a time, four partial sums
      const float2 nm2 = make_float2(-m_use, -m_use);
      float2 rs[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                      make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
      // P in the MMA's input type: two 16-bit or four e4m3 values a word
      uint32_t pk[L::kPCols];
#pragma unroll
      for (int cc = 0; cc < kBN; cc += 4) {
        const float2 x0 = __ffma2_rn(make_float2(sf[cc], sf[cc + 1]), c2, nm2);
        const float2 x1 = __ffma2_rn(make_float2(sf[cc + 2], sf[cc + 3]), c2, nm2);
        const float p0 = ptx::ex2_approx(x0.x);
        const float p1 = ptx::ex2_approx(x0.y);
        const float p2 = ptx::ex2_approx(x1.x);
        const float p3 = ptx::ex2_approx(x1.y);
        rs[(cc >> 1) & 3] = __fadd2_rn(rs[(cc >> 1) & 3], make_float2(p0, p1));
        rs[((cc >> 1) + 1) & 3] = __fadd2_rn(rs[((cc >> 1) + 1) & 3], make_float2(p2, p3));
        if constexpr (kF8) {
          pk[cc / 4] = ptx::pack_e4m3x4(p0, p1, p2, p3);
        } else if constexpr (T == kBF16) {
          pk[cc / 2] = ptx::pack_bf16(p0, p1);
          pk[cc / 2 + 1] = ptx::pack_bf16(p2, p3);
        } else {
          pk[cc / 2] = ptx::pack_f16(p0, p1);
          pk[cc / 2 + 1] = ptx::pack_f16(p2, p3);
        }
      }
      // O_i += P_i V_{j-1} must be complete before P_i is overwritten and
      // before O_i is rescaled.
      if (j > 0) {
        if (!wait_phase(bar(L::bODone + i), (j - 1) & 1, abort_flag, p)) { ok = false; break; }
        ptx::tc_fence_after();
      }
      if constexpr (kWideLdSt) {
        ptx::tmem_st64(tP, &pk[0]);
      } else {
#pragma unroll
        for (int cc = 0; cc < L::kPCols; cc += 32)
          ptx::tmem_st32(tP + cc, *reinterpret_cast<uint32_t(*)[32]>(&pk[cc]));
      }
      if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
        const float2 a2 = make_float2(alpha, alpha);
#pragma unroll
        for (int cc = 0; cc < D / 32; ++cc) {
          uint32_t o[32];
          ptx::tmem_ld32(tO + cc * 32, o);
          ptx::tmem_wait_ld();
          ptx::reg_fence32(o);
#pragma unroll
          for (int t = 0; t < 32; t += 2) {
            const float2 v2 = __fmul2_rn(make_float2(__uint_as_float(o[t]),
                                                     __uint_as_float(o[t + 1])), a2);
            o[t] = __float_as_uint(v2.x);
            o[t + 1] = __float_as_uint(v2.y);
          }
          ptx::tmem_st32(tO + cc * 32, o);
        }
      }
      ptx::tmem_wait_st();
      ptx::tc_fence_before();
      if constexpr (kWarpArrive) {
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(bar(L::bPFull + (L::kMerged ? 0 : i)));
      } else {
        ptx::mbar_arrive(bar(L::bPFull + (L::kMerged ? 0 : i)));
      }
      const float2 r01 = __fadd2_rn(rs[0], rs[1]);
      const float2 r23 = __fadd2_rn(rs[2], rs[3]);
      l = l * alpha + ((r01.x + r01.y) + (r23.x + r23.y));
      if (m_new != -CUDART_INF_F) m = m_use;
    }

    if constexpr (kSkip) {
      // Blocks nb_i .. nb-1 lie wholly past this tile's diagonal.  The merged
      // "scores read" and "P written" barriers count both warpgroups, so this
      // one still arrives on each, once the previous block's phase is
      // complete (so that the arrivals count toward this block's phase).
      for (int j = nb_i; ok && j < nb; ++j) {
        if (!wait_phase(bar(L::bSFree), (j - 1) & 1, abort_flag, p)) { ok = false; break; }
        ptx::mbar_arrive(bar(L::bSFree));
        if (!wait_phase(bar(L::bPFull), (j - 1) & 1, abort_flag, p)) { ok = false; break; }
        ptx::mbar_arrive(bar(L::bPFull));
      }
    }

    // ---- epilogue: O / l and LSE
    if (ok && nb_i > 0) ok = wait_phase(bar(L::bODone + i), (nb_i - 1) & 1, abort_flag, p);
    // One query tile: each warp stages its 32 rows of O in the tile's Q region
    // (free once the tile's MMAs are done: the last product's commit covers
    // every earlier MMA), XOR-swizzled by row so that neither the row-wise
    // writes nor the chunk-wise reads conflict on banks, then stores them 512
    // contiguous bytes an instruction instead of 16 bytes to each of 32 rows
    // (measured: +2 to +4.5 % at N = 512..2048; in the two-tile kernels the
    // same code cost 5 % at N = 8192 through the main loop's code generation).
    constexpr bool kStageO = Q == 1;
    constexpr int kORowBytes = D * 2;
    static_assert(!kStageO || 128 * kORowBytes <= L::kBars, "staged O fits below the barriers");
    if constexpr (kStageO) ok = __all_sync(0xffffffffu, ok);   // the staged store is warp-wide
    if (ok) {
      ptx::tc_fence_after();
      const bool valid = row < p.Nq;
      const float inv = l > 0.f ? p.o_scale / l : 0.f;
      const size_t orow = (size_t)bh * (size_t)p.Nq + (size_t)row;
      uint16_t *optr = reinterpret_cast<uint16_t *>(p.o) + orow * D;
      uint8_t *stage = smem + L::kQ + (warp & 3) * 32 * kORowBytes;
#pragma unroll
      for (int cc = 0; cc < D / 32; ++cc) {
        uint32_t o[32];
        if (nb_i > 0) {
          ptx::tmem_ld32(tO + cc * 32, o);
          ptx::tmem_wait_ld();
          ptx::reg_fence32(o);
        } else {
#pragma unroll
          for (int t = 0; t < 32; ++t) o[t] = 0u;
        }
        uint32_t w[16];
#pragma unroll
        for (int t = 0; t < 16; ++t) {
          const float a = __uint_as_float(o[2 * t]) * inv;
          const float b = __uint_as_float(o[2 * t + 1]) * inv;
          w[t] = kOutBF16 ? ptx::pack_bf16(a, b) : ptx::pack_f16(a, b);
        }
        if constexpr (kStageO) {
          uint8_t *srow = stage + lane * kORowBytes;
#pragma unroll
          for (int t = 0; t < 4; ++t)
            *reinterpret_cast<uint4 *>(srow + (((cc * 4 + t) ^ (lane & 7)) * 16)) =
                make_uint4(w[4 * t], w[4 * t + 1], w[4 * t + 2], w[4 * t + 3]);
        } else if (valid) {
          uint4 *dst = reinterpret_cast<uint4 *>(optr + cc * 32);
#pragma unroll
          for (int t = 0; t < 4; ++t)
            dst[t] = make_uint4(w[4 * t], w[4 * t + 1], w[4 * t + 2], w[4 * t + 3]);
        }
      }
      if constexpr (kStageO) {
        __syncwarp();
        constexpr int kChunksRow = kORowBytes / 16;
        const int row0 = q0 + (warp & 3) * 32;   // this warp's first row
        uint4 *obase = reinterpret_cast<uint4 *>(reinterpret_cast<uint16_t *>(p.o) +
                                                 ((size_t)bh * (size_t)p.Nq + (size_t)row0) * D);
#pragma unroll
        for (int k = 0; k < kChunksRow; ++k) {
          const int idx = k * 32 + lane;   // 16-byte chunk of the warp's rows
          const int rr = idx / kChunksRow, c = idx % kChunksRow;
          if (row0 + rr < p.Nq)
            obase[idx] = *reinterpret_cast<const uint4 *>(stage + rr * kORowBytes +
                                                          ((c ^ (rr & 7)) * 16));
        }
      }
      if (valid)
        p.lse[orow] = l > 0.f ? (m + log2f(l)) * 0.69314718055994531f : -CUDART_INF_F;
    }
  }

  // ---- teardown: all TMEM traffic of the CTA is complete before release
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, L::kTmem);
  }
}

}  // namespace fa
