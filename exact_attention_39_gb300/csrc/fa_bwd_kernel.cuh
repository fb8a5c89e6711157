// fa_bwd_kernel.cuh -- attention backward for sm_103a.
//
// For O = softmax(scale * Q K^T [mask]) V with logsumexp LSE and an upstream
// gradient dO:
//   P  = exp(scale * Q K^T - LSE)          (recomputed, never stored)
//   D  = rowsum(dO .* O)                   (one fp32 per query row)
//   dV = P^T dO,   dP = dO V^T,   dS = P .* (dP - D)
//   dQ = scale * dS K,   dK = scale * dS^T Q
// The benchmarks page lists the forward as recomputing the attention matrix
// instead of storing it ("0 MB (重计算)", Flash Attention 2 memory table);
// the backward recomputes P from Q, K and the stored LSE in the same way.
//
// Three kernels, no atomics:
//   fa_bwd_dot_kernel   -D for every query row, and -LSE in exp2 units, into
//                       the workspace, each head padded to whole 128-row
//                       blocks (0 and -inf on padding, so its probabilities
//                       are zero); negated so that the element-wise steps
//                       are packed two-wide adds and fused multiply-adds
//   fa_bwd_dq_kernel    one CTA per 128 query rows, looping over 64-key
//                       blocks: S = Q K^T and dP = dO V^T into TMEM, dS over
//                       dP, dQ += dS K (K read as the MN-major B operand)
//   fa_bwd_dkdv_kernel  one CTA per 128 keys, looping over 64-row query
//                       blocks: S^T = K Q^T and dP^T = V dO^T (keys on TMEM
//                       lanes), P^T and dS^T written over S^T (one store),
//                       dV += P^T dO, dK += dS^T Q
// Both main kernels: warps 0-7 element-wise in two warpgroups (thread = TMEM
// lane; warpgroup h takes columns 32h .. 32h+31 of each 64-column block and
// half of the output columns), warp 8 TMA producer, warp 9 TMEM allocator
// and MMA issuer (the whole warp runs the loop and one elected lane issues:
// inside a branch of its own at D = 64, as a predicate on MMAs the whole
// warp executes at D = 128).
//
// Pipelining.  S and dP of a block live in one of kBuf TMEM buffers; the
// MMA thread issues the gradient product of block n and then, into the same
// buffer, the scores of block n + kBuf.  The tensor pipe runs one thread's
// MMAs in issue order, so the product has read P (or dS) before the next
// scores overwrite it, and an element-wise thread that sees block n + kBuf's
// scores complete knows that block n's product is done with its columns.
// While the element-wise warps work on block n the pipe has the products of
// the blocks in between to run; nothing waits on a round trip per block.
//
// The operand that stays fixed over a CTA's loop (Q and dO in the dQ kernel;
// K and V in the dK/dV kernel for D = 64) is copied once from shared memory
// into TMEM by the element-wise warps and read from there as the A operand:
// with both operands in shared memory an M = 128, N = 64 MMA is held to the
// shared-memory read rate (6 KB per MMA, 48 cycles instead of 32 on the
// GB300); with A in TMEM it runs at the tensor pipe's rate.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <type_traits>

#include "fa_fwd_kernel.cuh"

namespace fa {

constexpr int kBwdThreads = 320;
constexpr int kBwdLoadWarp = 8;
constexpr int kBwdMmaWarp = 9;
constexpr int kBwdEwThreads = 256;       // element-wise threads
constexpr int kBwdBlk = 64;              // inner block: query rows (dK/dV) or keys (dQ)
constexpr int kBwdHalf = kBwdBlk / 2;    // columns of a block per element-wise thread

struct BwdParams {
  const void *o, *dout;      // [BH, Nq, D]
  const float *lse;          // [BH, Nq]
  float *nlse2;              // -LSE * log2(e), -inf where no key is seen, [BH, n_pad] (workspace)
  float *ndsum;              // -D = -rowsum(dO .* O), [BH, n_pad] (workspace)
  int n_pad;                 // Nq rounded up to whole 128-row blocks
  void *dq, *dk, *dv;        // outputs
  int Nq, Nk;
  int n_qblk, n_kblk;        // ceil(Nq / 128), ceil(Nk / 128)
  int causal;
  float c;                   // scale * log2(e)
  float scale;
  unsigned long long timeout_ns;
  unsigned *status;
};

// ---------------------------------------------------------------- D
// Eight lanes per padded row, each with D/8 consecutive elements (16-byte
// loads); lane 0 also converts the row's LSE to exp2 units.
template <int D, int T>
__global__ void __launch_bounds__(256)
    fa_bwd_dot_kernel(const BwdParams p, long long rows_pad) {
  const long long gid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const long long prow = gid >> 3;                 // padded row
  const int part = (int)(gid & 7);
  const long long bh = prow / p.n_pad;
  const int i = (int)(prow - bh * p.n_pad);
  const bool valid = prow < rows_pad && i < p.Nq;
  const long long row = bh * p.Nq + i;             // row of o, dout, lse
  float acc = 0.f;
  if (valid) {
    const uint4 *o = reinterpret_cast<const uint4 *>(
        reinterpret_cast<const uint16_t *>(p.o) + row * D + part * (D / 8));
    const uint4 *g = reinterpret_cast<const uint4 *>(
        reinterpret_cast<const uint16_t *>(p.dout) + row * D + part * (D / 8));
#pragma unroll
    for (int c = 0; c < D / 64; ++c) {
      const uint4 a = o[c], b = g[c];
      const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, bw[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        float2 fa2, fb2;
        if constexpr (T == kBF16) {
          fa2 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&aw[t]));
          fb2 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&bw[t]));
        } else {
          fa2 = __half22float2(*reinterpret_cast<const __half2 *>(&aw[t]));
          fb2 = __half22float2(*reinterpret_cast<const __half2 *>(&bw[t]));
        }
        acc = fmaf(fa2.x, fb2.x, acc);
        acc = fmaf(fa2.y, fb2.y, acc);
      }
    }
  }
  acc += __shfl_xor_sync(0xffffffffu, acc, 1);
  acc += __shfl_xor_sync(0xffffffffu, acc, 2);
  acc += __shfl_xor_sync(0xffffffffu, acc, 4);
  if (prow < rows_pad && part == 0) {
    float nl2 = -CUDART_INF_F;
    if (valid) {
      // a row that sees no key has LSE = -inf: its probabilities are zero
      const float lse = p.lse[row];
      nl2 = lse == -CUDART_INF_F ? -CUDART_INF_F : -lse * 1.4426950408889634f;
    }
    p.nlse2[prow] = nl2;
    p.ndsum[prow] = valid ? -acc : 0.f;
  }
}


// ---------------------------------------------------------------- layouts
// A 64-row block tile (Q and dO blocks of the dK/dV kernel, K and V blocks
// of the dQ kernel): the same 128-byte-swizzled chunks as a 128-row tile,
// each chunk kBwdBlk rows high.
template <int D, int T>
struct BlkTile {
  using F = Layout<D, T>;
  static constexpr int kChunkBytes = kBwdBlk * F::kSwz;
  static constexpr int kBytes = F::kChunks * kChunkBytes;
};

template <int D, int T>
struct BwdQLayout {
  using F = Layout<D, T>;
  using H = BlkTile<D, T>;
  static constexpr int kTile = F::kTileBytes;            // Q, dO: 128 rows
  static constexpr int kStages = D == 64 ? 8 : 4;        // K, V block ring
  static constexpr int kBuf = D == 64 ? 3 : 2;           // S, dP buffers in TMEM
  static constexpr int kQ = 0;
  static constexpr int kdO = kTile;
  static constexpr int kRing = 2 * kTile;
  static constexpr int kStageBytes = 2 * H::kBytes;      // K block, V block
  static constexpr int kBars = kRing + kStages * kStageBytes;
  // D = 128: the whole MMA warp executes each MMA, predicated on the issuing
  // lane (see ptx::mma_ts_if); D = 64: the issuing lane alone, in a branch.
  // Measured on the GB300 per kernel and head dim: predicated +4 % (dQ) and
  // +5 % (dK/dV) at D = 128, -4 % and -3 % at D = 64.
  static constexpr bool kPredIssue = D == 128;
  static constexpr int bQFull = 0;
  static constexpr int bKVFull = 1;                      // [stages]
  static constexpr int bKVEmpty = bKVFull + kStages;     // [stages]
  static constexpr int bSFull = bKVEmpty + kStages;      // [kBuf]: S and dP done
  static constexpr int bDSFull = bSFull + kBuf;          // [kBuf]: dS written
  static constexpr int bAFull = bDSFull + kBuf;          // Q, dO copied into TMEM
  static constexpr int bGDone = bAFull + 1;              // every dQ product done
  static constexpr int bDrain = bGDone + 1;
  static constexpr int kNumBars = bDrain + 1;
  static constexpr int kMisc = kBars + kNumBars * 8;
  static constexpr int kAlloc = kMisc + 16 + 1024;
  __host__ __device__ static constexpr int stage(int s) { return kRing + s * kStageBytes; }
  // TMEM columns: S(b), dP(b) (dS over the first columns of each half),
  // the dQ accumulator, then Q and dO as 16-bit pairs
  __host__ __device__ static constexpr uint32_t tS(int b) { return 64u * b; }
  __host__ __device__ static constexpr uint32_t tdP(int b) { return 64u * (kBuf + b); }
  static constexpr uint32_t tdQ = 128u * kBuf;
  static constexpr uint32_t tQa = tdQ + D;
  static constexpr uint32_t tdOa = tQa + D / 2;
  static_assert(tdOa + D / 2 <= (uint32_t)kTmemCols, "TMEM columns");
  static_assert(kAlloc <= 227 * 1024, "shared memory");
};

template <int D, int T>
struct BwdKVLayout {
  using F = Layout<D, T>;
  using H = BlkTile<D, T>;
  // D = 64: K and V as TMEM A operands (every product an A-in-TMEM MMA).
  // D = 128: the accumulators take half of TMEM and K, V stay in shared
  // memory (S^T and dP^T then read both operands from there).
  static constexpr bool kATmem = D == 64;
  static constexpr int kTile = F::kTileBytes;            // K, V: 128 rows
  // Q block, dO block, then 64 floats of -LSE and 64 of -D (1 KB-aligned)
  static constexpr int kStageBytes = 2 * H::kBytes + 1024;
  static constexpr int kStages = D == 64 ? 8 : 4;
  static constexpr int kBuf = 2;
  static constexpr int kK = 0, kV = kTile;
  static constexpr int kStage0 = 2 * kTile;
  static constexpr int kBars = kStage0 + kStages * kStageBytes;
  static constexpr bool kPredIssue = D == 128;   // as in the dQ kernel
  static constexpr int bKVFull = 0;
  static constexpr int bQFull = 1;                       // [stages]
  static constexpr int bQEmpty = bQFull + kStages;       // [stages]
  static constexpr int bSFull = bQEmpty + kStages;       // [kBuf]: S^T, dP^T done
  static constexpr int bPFull = bSFull + kBuf;           // [kBuf]: P^T, dS^T written
  static constexpr int bAFull = bPFull + kBuf;           // K, V copied into TMEM
  static constexpr int bGDone = bAFull + 1;              // every dV, dK product done
  static constexpr int bDrain = bGDone + 1;
  static constexpr int kNumBars = bDrain + 1;
  static constexpr int kMisc = kBars + kNumBars * 8;
  static constexpr int kAlloc = kMisc + 16 + 1024;
  __host__ __device__ static constexpr int stage(int s) { return kStage0 + s * kStageBytes; }
  __host__ __device__ static constexpr uint32_t tS(int b) { return 64u * b; }
  __host__ __device__ static constexpr uint32_t tdP(int b) { return 64u * (kBuf + b); }
  static constexpr uint32_t tdV = 128u * kBuf;
  static constexpr uint32_t tdK = tdV + D;
  static constexpr uint32_t tKa = tdK + D;               // kATmem only
  static constexpr uint32_t tVa = tKa + D / 2;
  static_assert((kATmem ? tVa + D / 2 : tdK + D) <= (uint32_t)kTmemCols, "TMEM columns");
  static_assert(kAlloc <= 227 * 1024, "shared memory");
};

// 16-bit pair packing of the element type
template <int T>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  return T == kBF16 ? ptx::pack_bf16(lo, hi) : ptx::pack_f16(lo, hi);
}

// MMA issue in one of two forms: kPred, the whole warp executes the
// instruction predicated on `issue`; otherwise the caller is already inside
// the issuing lane's branch and the instruction is plain.
template <bool kPred>
__device__ __forceinline__ void mma_ts_sel(uint32_t d, uint32_t a, uint64_t b, uint32_t idesc,
                                           uint32_t acc, uint32_t issue) {
  if constexpr (kPred) ptx::mma_ts_if(d, a, b, idesc, acc, issue);
  else ptx::mma_ts(d, a, b, idesc, acc);
}
template <bool kPred>
__device__ __forceinline__ void mma_ss_sel(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                           uint32_t acc, uint32_t issue) {
  if constexpr (kPred) ptx::mma_ss_if(d, a, b, idesc, acc, issue);
  else ptx::mma_ss(d, a, b, idesc, acc);
}
template <bool kPred>
__device__ __forceinline__ void mma_commit_sel(uint32_t bar, uint32_t issue) {
  if constexpr (kPred) ptx::mma_commit_if(bar, issue);
  else ptx::mma_commit(bar);
}

// Shared set-up of both main kernels: 1 KB-aligned shared memory, TMEM
// allocation by the MMA warp, barrier initialisation by thread 0.
struct BwdSmem {
  uint32_t sbase;
  uint8_t *smem;
};

__device__ __forceinline__ BwdSmem bwd_smem(uint8_t *smem_raw) {
  const uint32_t raw = ptx::smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  return {sbase, smem_raw + (sbase - raw)};
}

// Copies row r of a 128-row tile (chunks of 128 rows x 128 bytes in the TMA
// 128-byte swizzle) into the calling thread's TMEM lane: D/2 columns of
// 16-bit pairs, element 2c in the low half of column c -- the layout of an
// A operand in TMEM.
template <int D, int T>
__device__ __forceinline__ void tile_row_to_tmem(const uint8_t *tile, int r, uint32_t taddr) {
  using F = Layout<D, T>;
  static_assert(F::kSwz == 128, "128-byte rows");
#pragma unroll
  for (int c = 0; c < F::kChunks; ++c) {
    uint32_t w[32];
    const uint8_t *row = tile + c * F::kChunkBytes + r * 128;
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const uint4 x = *reinterpret_cast<const uint4 *>(row + ((u ^ (r & 7)) << 4));
      w[4 * u] = x.x;
      w[4 * u + 1] = x.y;
      w[4 * u + 2] = x.z;
      w[4 * u + 3] = x.w;
    }
    ptx::tmem_st32(taddr + 32u * c, w);
  }
}

// The A columns of K step kk (16 elements) of a 64-column block whose two
// halves (32 elements, 16 columns of pairs) sit at +0 and +32.
__device__ __forceinline__ constexpr uint32_t half_cols(int kk) {
  return (uint32_t)((kk >> 1) * 32 + (kk & 1) * 8);
}

// ---------------------------------------------------------------- dQ
template <int D, int T>
__global__ void __launch_bounds__(kBwdThreads, 1)
    fa_bwd_dq_kernel(const __grid_constant__ CUtensorMap tmQ,     // 128-row boxes
                     const __grid_constant__ CUtensorMap tmK,     // 64-row boxes
                     const __grid_constant__ CUtensorMap tmV,     // 64-row boxes
                     const __grid_constant__ CUtensorMap tmdO,    // 128-row boxes
                     const BwdParams p) {
  using L = BwdQLayout<D, T>;
  using F = typename L::F;
  using H = typename L::H;
  using E = Elem<T>;
  constexpr int kBuf = L::kBuf;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const BwdSmem sm = bwd_smem(smem_raw);
  const uint32_t sbase = sm.sbase;
  const uint32_t bars = sbase + L::kBars;
  auto bar = [&](int idx) -> uint32_t { return bars + 8u * (uint32_t)idx; };
  volatile uint32_t *tmem_slot = reinterpret_cast<volatile uint32_t *>(sm.smem + L::kMisc);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(sm.smem + L::kMisc + 4);
  const int warp = threadIdx.x >> 5;

  const int bh = blockIdx.x / p.n_qblk;
  int qb = blockIdx.x % p.n_qblk;
  if (p.causal) qb = p.n_qblk - 1 - qb;                  // longest first
  const int q0 = qb * kBM;
  int kv_end = p.Nk;
  if (p.causal) kv_end = min(p.Nk, q0 + kBM + (p.Nk - p.Nq));
  const int nb = kv_end > 0 ? (kv_end + kBwdBlk - 1) / kBwdBlk : 0;   // 64-key blocks

  if (warp == kBwdMmaWarp) {
    ptx::tmem_alloc(sbase + L::kMisc, kTmemCols);
    ptx::tmem_relinquish();
  }
  if (threadIdx.x == 0) {
    ptx::mbar_init(bar(L::bQFull), 1);
    for (int s = 0; s < L::kStages; ++s) {
      ptx::mbar_init(bar(L::bKVFull + s), 1);
      ptx::mbar_init(bar(L::bKVEmpty + s), 1);
    }
    for (int b = 0; b < kBuf; ++b) {
      ptx::mbar_init(bar(L::bSFull + b), 1);
      ptx::mbar_init(bar(L::bDSFull + b), kBwdEwThreads);
    }
    ptx::mbar_init(bar(L::bAFull), kBwdEwThreads);
    ptx::mbar_init(bar(L::bGDone), 1);
    ptx::mbar_init(bar(L::bDrain), 1);
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == kBwdLoadWarp) {
    // ================================================= TMA producer
    if (nb > 0) {
      const bool leader = ptx::elect_one();
      const uint64_t pol_q = ptx::policy_evict_first();
      const uint64_t pol_kv = ptx::policy_evict_last();
      if (leader) {
        ptx::mbar_arrive_expect_tx(bar(L::bQFull), 2 * L::kTile);
        for (int c = 0; c < F::kChunks; ++c) {
          ptx::tma_load_3d(sbase + L::kQ + c * F::kChunkBytes, &tmQ, bar(L::bQFull),
                           c * F::kChunkElems, q0, bh, pol_q);
          ptx::tma_load_3d(sbase + L::kdO + c * F::kChunkBytes, &tmdO, bar(L::bQFull),
                           c * F::kChunkElems, q0, bh, pol_q);
        }
      }
      int issued = 0;
      for (int j = 0; j < nb; ++j) {
        const int st = j % L::kStages, use = j / L::kStages;
        if (use > 0 && !wait_warp(bar(L::bKVEmpty + st), (use - 1) & 1, abort_flag, p)) break;
        if (leader) {
          const uint32_t sa = sbase + L::stage(st);
          ptx::mbar_arrive_expect_tx(bar(L::bKVFull + st), 2 * H::kBytes);
          for (int c = 0; c < F::kChunks; ++c) {
            ptx::tma_load_3d(sa + c * H::kChunkBytes, &tmK, bar(L::bKVFull + st),
                             c * F::kChunkElems, j * kBwdBlk, bh, pol_kv);
            ptx::tma_load_3d(sa + H::kBytes + c * H::kChunkBytes, &tmV, bar(L::bKVFull + st),
                             c * F::kChunkElems, j * kBwdBlk, bh, pol_kv);
          }
        }
        issued = j + 1;
      }
      wait_drain(bar(L::bQFull), 0, p);
      for (int j = issued - L::kStages; j < issued; ++j) {
        if (j < 0) continue;
        wait_drain(bar(L::bKVFull + j % L::kStages), (uint32_t)(j / L::kStages) & 1u, p);
      }
    }
  } else if (warp == kBwdMmaWarp) {
    // ================================================= MMA issuer
    if (nb > 0) {
      const bool leader = ptx::elect_one();
      const uint32_t iss = leader ? 1u : 0u;   // the issuing lane (predicated issue)
      constexpr bool kP = L::kPredIssue;
      constexpr uint32_t idesc_s = make_idesc(kBM, kBwdBlk, E::kFmt, false);
      constexpr uint32_t idesc_q = make_idesc(kBM, D, E::kFmt, true);
      const uint64_t dk0 = make_sdesc(sbase + L::stage(0), 16, F::kSBO, F::kSwzMode);
      const uint64_t dv0 = make_sdesc(sbase + L::stage(0) + H::kBytes, 16, F::kSBO, F::kSwzMode);
      const uint64_t dkmn0 = make_sdesc(sbase + L::stage(0), H::kChunkBytes, F::kSBO, F::kSwzMode);
      // S(b) = Q K_st^T and dP(b) = dO V_st^T, then a commit on s_full[b]
      auto issue_s = [&](int st, int b) {
        const uint64_t so = (uint64_t)((st * L::kStageBytes) >> 4);
        if (kP || leader) {
#pragma unroll
          for (int kk = 0; kk < D / E::kMmaK; ++kk) {
            const uint32_t off = ((kk >> 2) * H::kChunkBytes + (kk & 3) * 32) >> 4;
            mma_ts_sel<kP>(tmem + L::tS(b), tmem + L::tQa + kk * 8, dk0 + so + off, idesc_s,
                           kk > 0, iss);
          }
#pragma unroll
          for (int kk = 0; kk < D / E::kMmaK; ++kk) {
            const uint32_t off = ((kk >> 2) * H::kChunkBytes + (kk & 3) * 32) >> 4;
            mma_ts_sel<kP>(tmem + L::tdP(b), tmem + L::tdOa + kk * 8, dv0 + so + off, idesc_s,
                           kk > 0, iss);
          }
          mma_commit_sel<kP>(bar(L::bSFull + b), iss);
        }
      };
      // dQ (+)= dS(b) K_st, then a commit on kv_empty[st]
      auto issue_dq = [&](int st, int b, bool acc) {
        const uint64_t so = (uint64_t)((st * L::kStageBytes) >> 4);
        if (kP || leader) {
#pragma unroll
          for (int kk = 0; kk < kBwdBlk / E::kMmaK; ++kk)
            mma_ts_sel<kP>(tmem + L::tdQ, tmem + L::tdP(b) + half_cols(kk),
                           dkmn0 + so + (uint64_t)((kk * E::kMmaK * F::kSwz) >> 4), idesc_q,
                           (acc || kk > 0) ? 1u : 0u, iss);
          mma_commit_sel<kP>(bar(L::bKVEmpty + st), iss);
        }
      };
      bool ok = wait_warp(bar(L::bAFull), 0, abort_flag, p);
      for (int j = 0; ok && j < kBuf && j < nb; ++j) {
        if (!wait_warp(bar(L::bKVFull + j), 0, abort_flag, p)) { ok = false; break; }
        ptx::tc_fence_after();
        issue_s(j, j);
      }
      for (int j = 0; ok && j < nb; ++j) {
        const int b = j % kBuf;
        if (!wait_warp(bar(L::bDSFull + b), (j / kBuf) & 1, abort_flag, p)) { ok = false; break; }
        ptx::tc_fence_after();
        issue_dq(j % L::kStages, b, j > 0);
        const int m = j + kBuf;   // into the buffer just read
        if (m < nb) {
          const int st = m % L::kStages;
          if (!wait_warp(bar(L::bKVFull + st), (m / L::kStages) & 1, abort_flag, p)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          issue_s(st, b);
        }
      }
      if (ok && leader) ptx::mma_commit(bar(L::bGDone));
      if (leader) ptx::mma_commit(bar(L::bDrain));
      wait_drain(bar(L::bDrain), 0, p);
    }
  } else {
    // ================================================= element-wise warps
    const int h = warp >> 2;                        // column half
    const int r = (warp & 3) * 32 + (threadIdx.x & 31);   // row = TMEM lane
    const int row = q0 + r;
    const bool valid = row < p.Nq;
    const uint32_t lane_off = (uint32_t)(32 * (warp & 3)) << 16;
    const size_t grow = (size_t)bh * (size_t)p.Nq + (size_t)row;
    const size_t prow = (size_t)bh * (size_t)p.n_pad + (size_t)row;   // row < n_pad
    const float nl2 = p.nlse2[prow], nd = p.ndsum[prow];
    const float2 nl2x2 = make_float2(nl2, nl2), ndx2 = make_float2(nd, nd);
    const int key_lim = p.causal ? min(p.Nk, row + 1 + (p.Nk - p.Nq)) : p.Nk;
    const float c = p.c;
    const float2 c2 = make_float2(c, c);
    bool ok = true;
    if (nb > 0) {
      // this thread's row of Q (first warpgroup) or dO (second) into TMEM
      ok = wait_warp(bar(L::bQFull), 0, abort_flag, p);
      if (ok) {
        tile_row_to_tmem<D, T>(sm.smem + (h == 0 ? L::kQ : L::kdO), r,
                               tmem + lane_off + (h == 0 ? L::tQa : L::tdOa));
        ptx::tmem_wait_st();
        ptx::tc_fence_before();
        ptx::mbar_arrive(bar(L::bAFull));
      }
    }
    for (int j = 0; ok && j < nb; ++j) {
      const int b = j % kBuf;
      if (!wait_warp(bar(L::bSFull + b), (j / kBuf) & 1, abort_flag, p)) { ok = false; break; }
      ptx::tc_fence_after();
      const uint32_t cs = tmem + lane_off + L::tS(b) + h * kBwdHalf;
      const uint32_t cdp = tmem + lane_off + L::tdP(b) + h * kBwdHalf;
      uint32_t s[kBwdHalf], dp[kBwdHalf];
      ptx::tmem_ld32(cs, s);
      ptx::tmem_ld32(cdp, dp);
      ptx::tmem_wait_ld();
      ptx::reg_fence32(s);
      ptx::reg_fence32(dp);
      const int lim = key_lim - j * kBwdBlk - h * kBwdHalf;   // this half's columns >= lim: masked
      uint32_t pk[kBwdHalf / 2];
      // dS = P .* (dP - D), two columns at a time; the mask test only on
      // blocks where some row of the warp has masked columns
      auto ds_block = [&](auto mask_tag) {
        constexpr bool kMask = decltype(mask_tag)::value;
#pragma unroll
        for (int t = 0; t < kBwdHalf; t += 2) {
          const float2 x = __ffma2_rn(make_float2(__uint_as_float(s[t]), __uint_as_float(s[t + 1])),
                                      c2, nl2x2);
          float2 pr = make_float2(ptx::ex2_approx(x.x), ptx::ex2_approx(x.y));
          if (kMask) {
            if (t >= lim) pr.x = 0.f;
            if (t + 1 >= lim) pr.y = 0.f;
          }
          const float2 g = __fadd2_rn(make_float2(__uint_as_float(dp[t]), __uint_as_float(dp[t + 1])),
                                      ndx2);
          const float2 ds = __fmul2_rn(pr, g);
          pk[t / 2] = pack2<T>(ds.x, ds.y);
        }
      };
      if (__any_sync(0xffffffffu, lim < kBwdHalf))
        ds_block(std::true_type{});
      else
        ds_block(std::false_type{});
      // dS over the first 16 columns of this half of dP(b), which only this
      // thread has read
      ptx::tmem_st16(cdp, pk);
      ptx::tmem_wait_st();
      ptx::tc_fence_before();
      ptx::mbar_arrive(bar(L::bDSFull + b));
    }
    // ---- epilogue: dQ = scale * (dS K), this half's columns
    if (ok && nb > 0) ok = wait_warp(bar(L::bGDone), 0, abort_flag, p);
    if (ok) {
      ptx::tc_fence_after();
      uint16_t *out = reinterpret_cast<uint16_t *>(p.dq) + grow * D + h * (D / 2);
#pragma unroll
      for (int cc = 0; cc < D / 2; cc += 32) {
        uint32_t g[32];
        if (nb > 0) {
          ptx::tmem_ld32(tmem + lane_off + L::tdQ + h * (D / 2) + cc, g);
          ptx::tmem_wait_ld();
          ptx::reg_fence32(g);
        } else {
#pragma unroll
          for (int t = 0; t < 32; ++t) g[t] = 0u;
        }
        uint32_t w[16];
#pragma unroll
        for (int t = 0; t < 16; ++t)
          w[t] = pack2<T>(__uint_as_float(g[2 * t]) * p.scale,
                          __uint_as_float(g[2 * t + 1]) * p.scale);
        if (valid) {
          uint4 *dst = reinterpret_cast<uint4 *>(out + cc);
#pragma unroll
          for (int t = 0; t < 4; ++t)
            dst[t] = make_uint4(w[4 * t], w[4 * t + 1], w[4 * t + 2], w[4 * t + 3]);
        }
      }
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == kBwdMmaWarp) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kTmemCols);
  }
}

// ---------------------------------------------------------------- dK, dV
template <int D, int T>
__global__ void __launch_bounds__(kBwdThreads, 1)
    fa_bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tmQ,    // 64-row boxes
                       const __grid_constant__ CUtensorMap tmK,    // 128-row boxes
                       const __grid_constant__ CUtensorMap tmV,    // 128-row boxes
                       const __grid_constant__ CUtensorMap tmdO,   // 64-row boxes
                       const BwdParams p) {
  using L = BwdKVLayout<D, T>;
  using F = typename L::F;
  using H = typename L::H;
  using E = Elem<T>;
  constexpr int kBuf = L::kBuf;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const BwdSmem sm = bwd_smem(smem_raw);
  const uint32_t sbase = sm.sbase;
  const uint32_t bars = sbase + L::kBars;
  auto bar = [&](int idx) -> uint32_t { return bars + 8u * (uint32_t)idx; };
  volatile uint32_t *tmem_slot = reinterpret_cast<volatile uint32_t *>(sm.smem + L::kMisc);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(sm.smem + L::kMisc + 4);
  const int warp = threadIdx.x >> 5;

  const int bh = blockIdx.x / p.n_kblk;
  const int kb = blockIdx.x % p.n_kblk;      // causal: small kb has the most work
  const int k0 = kb * kBN;
  // 64-row query blocks whose rows see at least one of these keys
  const int n_qb = (p.Nq + kBwdBlk - 1) / kBwdBlk;
  int i_begin = 0;
  if (p.causal) {
    const int first_row = k0 - (p.Nk - p.Nq);     // first row that sees key k0
    i_begin = first_row > 0 ? first_row / kBwdBlk : 0;
  }
  const int nqb = n_qb > i_begin ? n_qb - i_begin : 0;

  if (warp == kBwdMmaWarp) {
    ptx::tmem_alloc(sbase + L::kMisc, kTmemCols);
    ptx::tmem_relinquish();
  }
  if (threadIdx.x == 0) {
    ptx::mbar_init(bar(L::bKVFull), 1);
    for (int s = 0; s < L::kStages; ++s) {
      ptx::mbar_init(bar(L::bQFull + s), 1);         // Q, dO blocks and LSE, D rows
      ptx::mbar_init(bar(L::bQEmpty + s), 1);
    }
    for (int b = 0; b < kBuf; ++b) {
      ptx::mbar_init(bar(L::bSFull + b), 1);
      ptx::mbar_init(bar(L::bPFull + b), kBwdEwThreads);
    }
    ptx::mbar_init(bar(L::bAFull), kBwdEwThreads);
    ptx::mbar_init(bar(L::bGDone), 1);
    ptx::mbar_init(bar(L::bDrain), 1);
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == kBwdLoadWarp) {
    // ================================================= producer
    if (nqb > 0) {
      const bool leader = ptx::elect_one();
      const uint64_t pol_kv = ptx::policy_evict_first();
      const uint64_t pol_q = ptx::policy_evict_last();
      if (leader) {
        ptx::mbar_arrive_expect_tx(bar(L::bKVFull), 2 * L::kTile);
        for (int c = 0; c < F::kChunks; ++c) {
          ptx::tma_load_3d(sbase + L::kK + c * F::kChunkBytes, &tmK, bar(L::bKVFull),
                           c * F::kChunkElems, k0, bh, pol_kv);
          ptx::tma_load_3d(sbase + L::kV + c * F::kChunkBytes, &tmV, bar(L::bKVFull),
                           c * F::kChunkElems, k0, bh, pol_kv);
        }
      }
      int issued = 0;
      for (int n = 0; n < nqb; ++n) {
        const int i = i_begin + n;
        const int st = n % L::kStages, use = n / L::kStages;
        if (use > 0 && !wait_warp(bar(L::bQEmpty + st), (use - 1) & 1, abort_flag, p)) break;
        const uint32_t sa = sbase + L::stage(st);
        if (leader) {
          ptx::mbar_arrive_expect_tx(bar(L::bQFull + st), 2 * H::kBytes + 2 * kBwdBlk * 4);
          for (int c = 0; c < F::kChunks; ++c) {
            ptx::tma_load_3d(sa + c * H::kChunkBytes, &tmQ, bar(L::bQFull + st),
                             c * F::kChunkElems, i * kBwdBlk, bh, pol_q);
            ptx::tma_load_3d(sa + H::kBytes + c * H::kChunkBytes, &tmdO, bar(L::bQFull + st),
                             c * F::kChunkElems, i * kBwdBlk, bh, pol_q);
          }
          // the block's 64 rows of -LSE (exp2 units) and -D: padded rows
          // (i * 64 + 64 <= n_pad)
          const size_t prow = (size_t)bh * (size_t)p.n_pad + (size_t)i * kBwdBlk;
          ptx::bulk_load(sa + 2 * H::kBytes, p.nlse2 + prow, kBwdBlk * 4, bar(L::bQFull + st),
                         pol_q);
          ptx::bulk_load(sa + 2 * H::kBytes + kBwdBlk * 4, p.ndsum + prow, kBwdBlk * 4,
                         bar(L::bQFull + st), pol_q);
        }
        issued = n + 1;
      }
      wait_drain(bar(L::bKVFull), 0, p);
      for (int n = issued - L::kStages; n < issued; ++n) {
        if (n < 0) continue;
        wait_drain(bar(L::bQFull + n % L::kStages), (uint32_t)(n / L::kStages) & 1u, p);
      }
    }
  } else if (warp == kBwdMmaWarp) {
    // ================================================= MMA issuer
    if (nqb > 0) {
      const bool leader = ptx::elect_one();
      const uint32_t iss = leader ? 1u : 0u;   // the issuing lane (predicated issue)
      constexpr bool kP = L::kPredIssue;
      constexpr uint32_t idesc_s = make_idesc(kBN, kBwdBlk, E::kFmt, false);
      constexpr uint32_t idesc_g = make_idesc(kBN, D, E::kFmt, true);
      const uint64_t dk = make_sdesc(sbase + L::kK, 16, F::kSBO, F::kSwzMode);
      const uint64_t dv = make_sdesc(sbase + L::kV, 16, F::kSBO, F::kSwzMode);
      const uint64_t dq0 = make_sdesc(sbase + L::stage(0), 16, F::kSBO, F::kSwzMode);
      const uint64_t ddo0 = make_sdesc(sbase + L::stage(0) + H::kBytes, 16, F::kSBO, F::kSwzMode);
      const uint64_t dqmn0 = make_sdesc(sbase + L::stage(0), H::kChunkBytes, F::kSBO, F::kSwzMode);
      const uint64_t ddomn0 = make_sdesc(sbase + L::stage(0) + H::kBytes, H::kChunkBytes, F::kSBO,
                                         F::kSwzMode);
      // S^T(b) = K Q_st^T and dP^T(b) = V dO_st^T, then a commit on s_full[b]
      auto issue_s = [&](int st, int b) {
        const uint64_t so = (uint64_t)((st * L::kStageBytes) >> 4);
        if (kP || leader) {
#pragma unroll
          for (int kk = 0; kk < D / E::kMmaK; ++kk) {
            const uint32_t ob = ((kk >> 2) * H::kChunkBytes + (kk & 3) * 32) >> 4;
            if constexpr (L::kATmem) {
              mma_ts_sel<kP>(tmem + L::tS(b), tmem + L::tKa + kk * 8, dq0 + so + ob, idesc_s,
                             kk > 0, iss);
            } else {
              const uint32_t oa = ((kk >> 2) * F::kChunkBytes + (kk & 3) * 32) >> 4;
              mma_ss_sel<kP>(tmem + L::tS(b), dk + oa, dq0 + so + ob, idesc_s, kk > 0, iss);
            }
          }
#pragma unroll
          for (int kk = 0; kk < D / E::kMmaK; ++kk) {
            const uint32_t ob = ((kk >> 2) * H::kChunkBytes + (kk & 3) * 32) >> 4;
            if constexpr (L::kATmem) {
              mma_ts_sel<kP>(tmem + L::tdP(b), tmem + L::tVa + kk * 8, ddo0 + so + ob, idesc_s,
                             kk > 0, iss);
            } else {
              const uint32_t oa = ((kk >> 2) * F::kChunkBytes + (kk & 3) * 32) >> 4;
              mma_ss_sel<kP>(tmem + L::tdP(b), dv + oa, ddo0 + so + ob, idesc_s, kk > 0, iss);
            }
          }
          mma_commit_sel<kP>(bar(L::bSFull + b), iss);
        }
      };
      // dV (+)= P^T(b) dO_st and dK (+)= dS^T(b) Q_st, then a commit on
      // q_empty[st]
      auto issue_g = [&](int st, int b, bool acc) {
        const uint64_t so = (uint64_t)((st * L::kStageBytes) >> 4);
        if (kP || leader) {
#pragma unroll
          for (int kk = 0; kk < kBwdBlk / E::kMmaK; ++kk)
            mma_ts_sel<kP>(tmem + L::tdV, tmem + L::tS(b) + half_cols(kk),
                           ddomn0 + so + (uint64_t)((kk * E::kMmaK * F::kSwz) >> 4), idesc_g,
                           (acc || kk > 0) ? 1u : 0u, iss);
#pragma unroll
          for (int kk = 0; kk < kBwdBlk / E::kMmaK; ++kk)
            mma_ts_sel<kP>(tmem + L::tdK, tmem + L::tS(b) + half_cols(kk) + 16,
                           dqmn0 + so + (uint64_t)((kk * E::kMmaK * F::kSwz) >> 4), idesc_g,
                           (acc || kk > 0) ? 1u : 0u, iss);
          mma_commit_sel<kP>(bar(L::bQEmpty + st), iss);
        }
      };
      bool ok = wait_warp(bar(L::bKVFull), 0, abort_flag, p) &&
                (!L::kATmem || wait_warp(bar(L::bAFull), 0, abort_flag, p));
      for (int n = 0; ok && n < kBuf && n < nqb; ++n) {
        if (!wait_warp(bar(L::bQFull + n), 0, abort_flag, p)) { ok = false; break; }
        ptx::tc_fence_after();
        issue_s(n, n);
      }
      for (int n = 0; ok && n < nqb; ++n) {
        const int b = n % kBuf;
        if (!wait_warp(bar(L::bPFull + b), (n / kBuf) & 1, abort_flag, p)) { ok = false; break; }
        ptx::tc_fence_after();
        issue_g(n % L::kStages, b, n > 0);
        const int m = n + kBuf;   // into the buffer just read
        if (m < nqb) {
          const int st = m % L::kStages;
          if (!wait_warp(bar(L::bQFull + st), (m / L::kStages) & 1, abort_flag, p)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          issue_s(st, b);
        }
      }
      if (ok && leader) ptx::mma_commit(bar(L::bGDone));
      if (leader) ptx::mma_commit(bar(L::bDrain));
      wait_drain(bar(L::bDrain), 0, p);
    }
  } else {
    // ================================================= element-wise warps
    const int h = warp >> 2;                        // query-column half
    const int r = (warp & 3) * 32 + (threadIdx.x & 31);   // key = TMEM lane
    const int key = k0 + r;
    const uint32_t lane_off = (uint32_t)(32 * (warp & 3)) << 16;
    const float c = p.c;
    const float2 c2 = make_float2(c, c);
    const int shift = p.Nk - p.Nq;                  // causal: key <= row + shift
    bool ok = true;
    if constexpr (L::kATmem) {
      if (nqb > 0) {
        // this thread's row of K (first warpgroup) or V (second) into TMEM
        ok = wait_warp(bar(L::bKVFull), 0, abort_flag, p);
        if (ok) {
          tile_row_to_tmem<D, T>(sm.smem + (h == 0 ? L::kK : L::kV), r,
                                 tmem + lane_off + (h == 0 ? L::tKa : L::tVa));
          ptx::tmem_wait_st();
          ptx::tc_fence_before();
          ptx::mbar_arrive(bar(L::bAFull));
        }
      }
    }
    for (int n = 0; ok && n < nqb; ++n) {
      const int i = i_begin + n;
      const int st = n % L::kStages;
      const int b = n % kBuf;
      if (!wait_warp(bar(L::bSFull + b), (n / kBuf) & 1, abort_flag, p) ||
          !wait_warp(bar(L::bQFull + st), (n / L::kStages) & 1, abort_flag, p)) {
        ok = false;
        break;
      }
      ptx::tc_fence_after();
      const float *lse_s = reinterpret_cast<const float *>(sm.smem + L::stage(st) + 2 * H::kBytes) +
                           h * kBwdHalf;
      const float *d_s = lse_s + kBwdBlk;
      // columns (query rows) of this half before `first` do not see the key
      const int first = p.causal ? key - shift - i * kBwdBlk - h * kBwdHalf : 0;
      const uint32_t cs = tmem + lane_off + L::tS(b) + h * kBwdHalf;
      const uint32_t cdp = tmem + lane_off + L::tdP(b) + h * kBwdHalf;
      uint32_t s[kBwdHalf], dp[kBwdHalf];
      ptx::tmem_ld32(cs, s);
      ptx::tmem_ld32(cdp, dp);
      ptx::tmem_wait_ld();
      ptx::reg_fence32(s);
      ptx::reg_fence32(dp);
      // P^T pairs in pk[0, 16), dS^T pairs in pk[16, 32): one 32-column store
      uint32_t pk[kBwdHalf];
      uint32_t *pkp = pk, *pkd = pk + kBwdHalf / 2;
      // P^T and dS^T = P^T .* (dP^T - D), two columns at a time (the
      // staged rows hold -LSE in exp2 units and -D); the causal test only on
      // blocks where some key of the warp has masked columns
      auto p_block = [&](auto mask_tag) {
        constexpr bool kMask = decltype(mask_tag)::value;
#pragma unroll
        for (int t = 0; t < kBwdHalf; t += 4) {
          const float4 l4 = *reinterpret_cast<const float4 *>(lse_s + t);
          const float4 d4 = *reinterpret_cast<const float4 *>(d_s + t);
          const float2 x0 = __ffma2_rn(make_float2(__uint_as_float(s[t]), __uint_as_float(s[t + 1])),
                                       c2, make_float2(l4.x, l4.y));
          const float2 x1 = __ffma2_rn(make_float2(__uint_as_float(s[t + 2]), __uint_as_float(s[t + 3])),
                                       c2, make_float2(l4.z, l4.w));
          float2 p0 = make_float2(ptx::ex2_approx(x0.x), ptx::ex2_approx(x0.y));
          float2 p1 = make_float2(ptx::ex2_approx(x1.x), ptx::ex2_approx(x1.y));
          if (kMask) {
            if (t < first) p0.x = 0.f;
            if (t + 1 < first) p0.y = 0.f;
            if (t + 2 < first) p1.x = 0.f;
            if (t + 3 < first) p1.y = 0.f;
          }
          const float2 g0 = __fadd2_rn(make_float2(__uint_as_float(dp[t]), __uint_as_float(dp[t + 1])),
                                       make_float2(d4.x, d4.y));
          const float2 g1 = __fadd2_rn(make_float2(__uint_as_float(dp[t + 2]), __uint_as_float(dp[t + 3])),
                                       make_float2(d4.z, d4.w));
          const float2 ds0 = __fmul2_rn(p0, g0), ds1 = __fmul2_rn(p1, g1);
          pkp[t / 2] = pack2<T>(p0.x, p0.y);
          pkp[t / 2 + 1] = pack2<T>(p1.x, p1.y);
          pkd[t / 2] = pack2<T>(ds0.x, ds0.y);
          pkd[t / 2 + 1] = pack2<T>(ds1.x, ds1.y);
        }
      };
      if (__any_sync(0xffffffffu, first > 0))
        p_block(std::true_type{});
      else
        p_block(std::false_type{});
      // P^T over the first 16 columns of this half of S^T(b) and dS^T over
      // the next 16: columns only this thread has read
      ptx::tmem_st32(cs, *reinterpret_cast<uint32_t(*)[32]>(&pk[0]));
      ptx::tmem_wait_st();
      ptx::tc_fence_before();
      ptx::mbar_arrive(bar(L::bPFull + b));
    }
    // ---- epilogue: dV and dK = scale * (dS^T Q), this half's columns
    if (ok && nqb > 0) ok = wait_warp(bar(L::bGDone), 0, abort_flag, p);
    if (ok) {
      ptx::tc_fence_after();
      const bool valid = key < p.Nk;
      const size_t gk = (size_t)bh * (size_t)p.Nk + (size_t)key;
#pragma unroll
      for (int which = 0; which < 2; ++which) {
        uint16_t *out = reinterpret_cast<uint16_t *>(which == 0 ? p.dv : p.dk) + gk * D +
                        h * (D / 2);
        const uint32_t tcol = (which == 0 ? L::tdV : L::tdK) + h * (D / 2);
        const float mul = which == 0 ? 1.f : p.scale;
#pragma unroll
        for (int cc = 0; cc < D / 2; cc += 32) {
          uint32_t g[32];
          if (nqb > 0) {
            ptx::tmem_ld32(tmem + lane_off + tcol + cc, g);
            ptx::tmem_wait_ld();
            ptx::reg_fence32(g);
          } else {
#pragma unroll
            for (int t = 0; t < 32; ++t) g[t] = 0u;
          }
          uint32_t w[16];
#pragma unroll
          for (int t = 0; t < 16; ++t)
            w[t] = pack2<T>(__uint_as_float(g[2 * t]) * mul,
                            __uint_as_float(g[2 * t + 1]) * mul);
          if (valid) {
            uint4 *dst = reinterpret_cast<uint4 *>(out + cc);
#pragma unroll
            for (int t = 0; t < 4; ++t)
              dst[t] = make_uint4(w[4 * t], w[4 * t + 1], w[4 * t + 2], w[4 * t + 3]);
          }
        }
      }
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == kBwdMmaWarp) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace fa
