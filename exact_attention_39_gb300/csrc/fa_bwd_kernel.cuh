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
//   fa_bwd_dq_kernel    one CTA per 128 query rows, looping over key blocks:
//                       S = Q K^T and dP = dO V^T into TMEM, dS to TMEM,
//                       dQ += dS K (K read as the MN-major B operand)
//   fa_bwd_dkdv_kernel  one CTA per 128 keys, looping over query blocks:
//                       S^T = K Q^T and dP^T = V dO^T (keys on TMEM lanes),
//                       P^T and dS^T to TMEM, dV += P^T dO, dK += dS^T Q
// Both main kernels: warps 0-7 element-wise in two warpgroups (thread = TMEM
// lane; warpgroup h takes columns 64h .. 64h+63 of each 128-column block and
// half of the output columns), warp 8 TMA producer, warp 9 TMEM allocator
// and MMA issuer.  No row reduction crosses the halves.
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
constexpr int kBwdHalf = 64;             // columns per element-wise thread

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
template <int D, int T>
struct BwdQLayout {
  using F = Layout<D, T>;
  static constexpr int kTile = F::kTileBytes;
  // D = 64: four stages, K and V of a stage on one barrier, and one "S and
  // dP read" wait per block gating both the next S, dP and the previous
  // block's dQ product (the loads then have two blocks of lead time).
  static constexpr bool kMerged = kTile <= 16384;
  static constexpr int kStages = kMerged ? 4 : 2;
  static constexpr int kQ = 0;                           // Q tile
  static constexpr int kdO = kTile;                      // dO tile
  static constexpr int kK = 2 * kTile;                   // K ring
  static constexpr int kV = kK + kStages * kTile;        // V ring
  static constexpr int kBars = kV + kStages * kTile;
  static constexpr int bQFull = 0;
  static constexpr int bKFull = 1;
  static constexpr int bVFull = bKFull + kStages;
  static constexpr int bKVEmpty = bVFull + kStages;
  static constexpr int bSFull = bKVEmpty + kStages;      // S and dP ready
  static constexpr int bSFree = bSFull + 1;              // S and dP read
  static constexpr int bDSFull = bSFree + 1;             // dS written
  static constexpr int bDQDone = bDSFull + 1;            // [2]: dQ MMA done
  static constexpr int bDrain = bDQDone + 2;
  static constexpr int kNumBars = bDrain + 1;
  static constexpr int kMisc = kBars + kNumBars * 8;
  static constexpr int kAlloc = kMisc + 16 + 1024;
  // TMEM columns
  static constexpr uint32_t tS = 0, tdP = 128, tdQ = 256;
  __host__ __device__ static constexpr uint32_t tdS(int b) { return 256 + D + 64 * b; }
};

template <int D, int T>
struct BwdKVLayout {
  using F = Layout<D, T>;
  static constexpr int kTile = F::kTileBytes;
  static constexpr int kStageBytes = 2 * kTile + 2 * kBM * 4;   // Q, dO, LSE, D
  static constexpr int kStages = kTile <= 16384 ? 4 : 2;
  static constexpr int kK = 0, kV = kTile;
  static constexpr int kStage0 = 2 * kTile;
  static constexpr int kBars = kStage0 + kStages * kStageBytes;
  static constexpr int bKVFull = 0;
  static constexpr int bQFull = 1;                       // [stages]
  static constexpr int bQEmpty = bQFull + kStages;       // [stages]
  static constexpr int bSFull = bQEmpty + kStages;       // S^T and dP^T ready
  static constexpr int bSFree = bSFull + 1;
  static constexpr int bPFull = bSFree + 1;              // P^T, dS^T written
  static constexpr int bPDone = bPFull + 1;              // dV, dK MMAs done
  static constexpr int bDrain = bPDone + 1;
  static constexpr int kNumBars = bDrain + 1;
  static constexpr int kMisc = kBars + kNumBars * 8;
  static constexpr int kAlloc = kMisc + 16 + 1024;
  // P^T and dS^T fit beside the accumulators for D = 64; for D = 128 they
  // overwrite the first 64 columns of S^T and dP^T once those are read.
  static constexpr bool kEarly = D == 64;
  static constexpr uint32_t tS = 0, tdP = 128, tdV = 256, tdK = 256 + D;
  static constexpr uint32_t tP = kEarly ? 384 : 0;
  static constexpr uint32_t tdS = kEarly ? 448 : 128;
  __host__ __device__ static constexpr int stage(int s) { return kStage0 + s * kStageBytes; }
};

// 16-bit pair packing of the element type
template <int T>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  return T == kBF16 ? ptx::pack_bf16(lo, hi) : ptx::pack_f16(lo, hi);
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

// ---------------------------------------------------------------- dQ
template <int D, int T>
__global__ void __launch_bounds__(kBwdThreads, 1)
    fa_bwd_dq_kernel(const __grid_constant__ CUtensorMap tmQ,
                     const __grid_constant__ CUtensorMap tmK,
                     const __grid_constant__ CUtensorMap tmV,
                     const __grid_constant__ CUtensorMap tmdO,
                     const BwdParams p) {
  using L = BwdQLayout<D, T>;
  using F = typename L::F;
  using E = Elem<T>;
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
  const int nb = kv_end > 0 ? (kv_end + kBN - 1) / kBN : 0;

  if (warp == kBwdMmaWarp) {
    ptx::tmem_alloc(sbase + L::kMisc, kTmemCols);
    ptx::tmem_relinquish();
  }
  if (threadIdx.x == 0) {
    ptx::mbar_init(bar(L::bQFull), 1);
    for (int s = 0; s < L::kStages; ++s) {
      ptx::mbar_init(bar(L::bKFull + s), 1);
      ptx::mbar_init(bar(L::bVFull + s), 1);
      ptx::mbar_init(bar(L::bKVEmpty + s), 1);
    }
    ptx::mbar_init(bar(L::bSFull), 1);
    ptx::mbar_init(bar(L::bSFree), kBwdEwThreads);
    ptx::mbar_init(bar(L::bDSFull), kBwdEwThreads);
    ptx::mbar_init(bar(L::bDQDone), 1);
    ptx::mbar_init(bar(L::bDQDone + 1), 1);
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
          const uint32_t vbar = bar(L::kMerged ? L::bKFull + st : L::bVFull + st);
          ptx::mbar_arrive_expect_tx(bar(L::bKFull + st), L::kMerged ? 2 * L::kTile : L::kTile);
          if (!L::kMerged) ptx::mbar_arrive_expect_tx(vbar, L::kTile);
          for (int c = 0; c < F::kChunks; ++c) {
            ptx::tma_load_3d(sbase + L::kK + st * L::kTile + c * F::kChunkBytes, &tmK,
                             bar(L::bKFull + st), c * F::kChunkElems, j * kBN, bh, pol_kv);
            ptx::tma_load_3d(sbase + L::kV + st * L::kTile + c * F::kChunkBytes, &tmV,
                             vbar, c * F::kChunkElems, j * kBN, bh, pol_kv);
          }
        }
        issued = j + 1;
      }
      wait_drain(bar(L::bQFull), 0, p);
      for (int j = issued - L::kStages; j < issued; ++j) {
        if (j < 0) continue;
        const int st = j % L::kStages;
        const uint32_t ph = (uint32_t)(j / L::kStages) & 1u;
        wait_drain(bar(L::bKFull + st), ph, p);
        if (!L::kMerged) wait_drain(bar(L::bVFull + st), ph, p);
      }
    }
  } else if (warp == kBwdMmaWarp) {
    // ================================================= MMA issuer
    if (nb > 0) {
      const bool leader = ptx::elect_one();
      constexpr uint32_t idesc_s = make_idesc(kBM, kBN, E::kFmt, false);
      constexpr uint32_t idesc_q = make_idesc(kBM, D, E::kFmt, true);
      const uint64_t dq_ = make_sdesc(sbase + L::kQ, 16, F::kSBO, F::kSwzMode);
      const uint64_t ddo = make_sdesc(sbase + L::kdO, 16, F::kSBO, F::kSwzMode);
      const uint64_t dk0 = make_sdesc(sbase + L::kK, 16, F::kSBO, F::kSwzMode);
      const uint64_t dv0 = make_sdesc(sbase + L::kV, 16, F::kSBO, F::kSwzMode);
      const uint64_t dkmn0 = make_sdesc(sbase + L::kK, F::kChunkBytes, F::kSBO, F::kSwzMode);
      // S = Q K_st^T and dP = dO V_st^T, then a commit on s_full
      auto issue_s = [&](int st) {
        const uint64_t dk = dk0 + (uint64_t)((st * L::kTile) >> 4);
        const uint64_t dv = dv0 + (uint64_t)((st * L::kTile) >> 4);
        if (leader) {
          // all of S's steps, then all of dP's (one accumulator at a time)
#pragma unroll
          for (int kk = 0; kk < D / E::kMmaK; ++kk) {
            const uint32_t off = ((kk >> 2) * F::kChunkBytes + (kk & 3) * 32) >> 4;
            ptx::mma_ss(tmem + L::tS, dq_ + off, dk + off, idesc_s, kk > 0);
          }
#pragma unroll
          for (int kk = 0; kk < D / E::kMmaK; ++kk) {
            const uint32_t off = ((kk >> 2) * F::kChunkBytes + (kk & 3) * 32) >> 4;
            ptx::mma_ss(tmem + L::tdP, ddo + off, dv + off, idesc_s, kk > 0);
          }
          ptx::mma_commit(bar(L::bSFull));
        }
      };
      // dQ (+)= dS_b K_st, then commits on dq_done[b] and kv_empty[st]
      auto issue_dq = [&](int st, int b, bool acc) {
        const uint64_t dk = dkmn0 + (uint64_t)((st * L::kTile) >> 4);
        if (leader) {
#pragma unroll
          for (int kk = 0; kk < kBN / E::kMmaK; ++kk)
            ptx::mma_ts(tmem + L::tdQ, tmem + L::tdS(b) + kk * 8,
                        dk + (uint64_t)((kk * E::kMmaK * F::kSwz) >> 4), idesc_q,
                        (acc || kk > 0) ? 1u : 0u);
          ptx::mma_commit(bar(L::bDQDone + b));
          ptx::mma_commit(bar(L::bKVEmpty + st));
        }
      };
      bool ok = wait_warp(bar(L::bQFull), 0, abort_flag, p) &&
                wait_warp(bar(L::bKFull), 0, abort_flag, p) &&
                (L::kMerged || wait_warp(bar(L::bVFull), 0, abort_flag, p));
      if (ok) {
        ptx::tc_fence_after();
        issue_s(0);
      }
      if constexpr (L::kMerged) {
        for (int j = 0; ok && j < nb; ++j) {
          const int st2 = (j + 1) % L::kStages;
          if (j + 1 < nb &&
              !wait_warp(bar(L::bKFull + st2), ((j + 1) / L::kStages) & 1, abort_flag, p)) {
            ok = false;
            break;
          }
          // S(j), dP(j) are in registers; dS(j-1) was written before that
          if (!wait_warp(bar(L::bSFree), j & 1, abort_flag, p)) { ok = false; break; }
          ptx::tc_fence_after();
          if (j + 1 < nb) issue_s(st2);
          if (j > 0) issue_dq((j - 1) % L::kStages, (j - 1) & 1, j > 1);
        }
        // the last block's dQ product once its dS is written
        if (ok && wait_warp(bar(L::bDSFull), 0, abort_flag, p)) {
          ptx::tc_fence_after();
          issue_dq((nb - 1) % L::kStages, (nb - 1) & 1, nb > 1);
        }
      }
      for (int j = 0; !L::kMerged && ok && j < nb; ++j) {
        const int st = j % L::kStages, st2 = (j + 1) % L::kStages;
        if (j + 1 < nb) {
          const uint32_t ph2 = ((j + 1) / L::kStages) & 1;
          if (!wait_warp(bar(L::bKFull + st2), ph2, abort_flag, p) ||
              !wait_warp(bar(L::bVFull + st2), ph2, abort_flag, p) ||
              !wait_warp(bar(L::bSFree), j & 1, abort_flag, p))
            break;
          ptx::tc_fence_after();
          issue_s(st2);
        }
        if (!wait_warp(bar(L::bDSFull), j & 1, abort_flag, p)) break;
        ptx::tc_fence_after();
        issue_dq(st, j & 1, j > 0);
      }
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
    for (int j = 0; j < nb; ++j) {
      const int b = j & 1;
      if (!wait_warp(bar(L::bSFull), j & 1, abort_flag, p)) { ok = false; break; }
      ptx::tc_fence_after();
      // S and dP of this half into registers first, so that the next
      // block's S and dP products overlap this block's element-wise work
      uint32_t s[kBwdHalf], dp[kBwdHalf];
#pragma unroll
      for (int cc = 0; cc < kBwdHalf; cc += 32) {
        ptx::tmem_ld32(tmem + lane_off + L::tS + h * kBwdHalf + cc,
                       *reinterpret_cast<uint32_t(*)[32]>(&s[cc]));
        ptx::tmem_ld32(tmem + lane_off + L::tdP + h * kBwdHalf + cc,
                       *reinterpret_cast<uint32_t(*)[32]>(&dp[cc]));
      }
      ptx::tmem_wait_ld();
#pragma unroll
      for (int cc = 0; cc < kBwdHalf; cc += 32) {
        ptx::reg_fence32(*reinterpret_cast<uint32_t(*)[32]>(&s[cc]));
        ptx::reg_fence32(*reinterpret_cast<uint32_t(*)[32]>(&dp[cc]));
      }
      ptx::tc_fence_before();
      ptx::mbar_arrive(bar(L::bSFree));
      const int lim = key_lim - j * kBN - h * kBwdHalf;   // this half's columns >= lim: masked
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
      if (j >= 2) {
        // dQ += dS_b K of two blocks back has finished reading dS_b
        if (!wait_warp(bar(L::bDQDone + b), ((j - 2) >> 1) & 1, abort_flag, p)) { ok = false; break; }
        ptx::tc_fence_after();
      }
      ptx::tmem_st32(tmem + lane_off + L::tdS(b) + h * (kBwdHalf / 2),
                     *reinterpret_cast<uint32_t(*)[32]>(&pk[0]));
      ptx::tmem_wait_st();
      ptx::tc_fence_before();
      // (merged: the MMA thread learns of dS(j) from the next S-read
      // arrival, so only the last block's dS is announced here)
      if (!L::kMerged || j == nb - 1) ptx::mbar_arrive(bar(L::bDSFull));
    }
    // ---- epilogue: dQ = scale * (dS K), this half's columns
    if (ok && nb > 0)
      ok = wait_warp(bar(L::bDQDone + ((nb - 1) & 1)), ((nb - 1) >> 1) & 1, abort_flag, p);
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
    fa_bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tmQ,
                       const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV,
                       const __grid_constant__ CUtensorMap tmdO,
                       const BwdParams p) {
  using L = BwdKVLayout<D, T>;
  using F = typename L::F;
  using E = Elem<T>;
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
  // query blocks whose rows see at least one of these keys
  int i_begin = 0;
  if (p.causal) {
    const int first_row = k0 - (p.Nk - p.Nq);     // first row that sees key k0
    i_begin = first_row > 0 ? first_row / kBM : 0;
  }
  const int nqb = p.n_qblk > i_begin ? p.n_qblk - i_begin : 0;

  if (warp == kBwdMmaWarp) {
    ptx::tmem_alloc(sbase + L::kMisc, kTmemCols);
    ptx::tmem_relinquish();
  }
  if (threadIdx.x == 0) {
    ptx::mbar_init(bar(L::bKVFull), 1);
    for (int s = 0; s < L::kStages; ++s) {
      ptx::mbar_init(bar(L::bQFull + s), 1);         // Q, dO tiles and LSE, D rows
      ptx::mbar_init(bar(L::bQEmpty + s), 1);
    }
    ptx::mbar_init(bar(L::bSFull), 1);
    ptx::mbar_init(bar(L::bSFree), kBwdEwThreads);
    ptx::mbar_init(bar(L::bPFull), kBwdEwThreads);
    ptx::mbar_init(bar(L::bPDone), 1);
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
          ptx::mbar_arrive_expect_tx(bar(L::bQFull + st), 2 * L::kTile + 2 * kBM * 4);
          for (int c = 0; c < F::kChunks; ++c) {
            ptx::tma_load_3d(sa + c * F::kChunkBytes, &tmQ, bar(L::bQFull + st),
                             c * F::kChunkElems, i * kBM, bh, pol_q);
            ptx::tma_load_3d(sa + L::kTile + c * F::kChunkBytes, &tmdO,
                             bar(L::bQFull + st), c * F::kChunkElems, i * kBM, bh, pol_q);
          }
          // the block's 128 rows of LSE (exp2 units) and D: whole padded rows
          const size_t prow = (size_t)bh * (size_t)p.n_pad + (size_t)i * kBM;
          ptx::bulk_load(sa + 2 * L::kTile, p.nlse2 + prow, kBM * 4, bar(L::bQFull + st), pol_q);
          ptx::bulk_load(sa + 2 * L::kTile + kBM * 4, p.ndsum + prow, kBM * 4,
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
      constexpr uint32_t idesc_s = make_idesc(kBN, kBM, E::kFmt, false);
      constexpr uint32_t idesc_g = make_idesc(kBN, D, E::kFmt, true);
      const uint64_t dk = make_sdesc(sbase + L::kK, 16, F::kSBO, F::kSwzMode);
      const uint64_t dv = make_sdesc(sbase + L::kV, 16, F::kSBO, F::kSwzMode);
      // S^T = K Q_st^T and dP^T = V dO_st^T, then a commit on s_full
      auto issue_s = [&](int st) {
        const uint32_t sa = sbase + L::stage(st);
        const uint64_t dq_ = make_sdesc(sa, 16, F::kSBO, F::kSwzMode);
        const uint64_t ddo = make_sdesc(sa + L::kTile, 16, F::kSBO, F::kSwzMode);
        if (leader) {
          // all of S^T's steps, then all of dP^T's
#pragma unroll
          for (int kk = 0; kk < D / E::kMmaK; ++kk) {
            const uint32_t off = ((kk >> 2) * F::kChunkBytes + (kk & 3) * 32) >> 4;
            ptx::mma_ss(tmem + L::tS, dk + off, dq_ + off, idesc_s, kk > 0);
          }
#pragma unroll
          for (int kk = 0; kk < D / E::kMmaK; ++kk) {
            const uint32_t off = ((kk >> 2) * F::kChunkBytes + (kk & 3) * 32) >> 4;
            ptx::mma_ss(tmem + L::tdP, dv + off, ddo + off, idesc_s, kk > 0);
          }
          ptx::mma_commit(bar(L::bSFull));
        }
      };
      // dV (+)= P^T dO_st and dK (+)= dS^T Q_st, then commits on p_done and
      // q_empty[st]
      auto issue_g = [&](int st, bool acc) {
        const uint32_t sa = sbase + L::stage(st);
        const uint64_t dq_mn = make_sdesc(sa, F::kChunkBytes, F::kSBO, F::kSwzMode);
        const uint64_t ddo_mn = make_sdesc(sa + L::kTile, F::kChunkBytes, F::kSBO, F::kSwzMode);
        if (leader) {
          // all of dV's steps, then all of dK's (one accumulator at a time)
#pragma unroll
          for (int kk = 0; kk < kBM / E::kMmaK; ++kk)
            ptx::mma_ts(tmem + L::tdV, tmem + L::tP + kk * 8,
                        ddo_mn + (uint64_t)((kk * E::kMmaK * F::kSwz) >> 4), idesc_g,
                        (acc || kk > 0) ? 1u : 0u);
#pragma unroll
          for (int kk = 0; kk < kBM / E::kMmaK; ++kk)
            ptx::mma_ts(tmem + L::tdK, tmem + L::tdS + kk * 8,
                        dq_mn + (uint64_t)((kk * E::kMmaK * F::kSwz) >> 4), idesc_g,
                        (acc || kk > 0) ? 1u : 0u);
          ptx::mma_commit(bar(L::bPDone));
          ptx::mma_commit(bar(L::bQEmpty + st));
        }
      };
      bool ok = wait_warp(bar(L::bKVFull), 0, abort_flag, p) &&
                wait_warp(bar(L::bQFull), 0, abort_flag, p);
      if (ok) {
        ptx::tc_fence_after();
        issue_s(0);
      }
      if constexpr (L::kEarly) {
        for (int n = 0; ok && n < nqb; ++n) {
          const int st2 = (n + 1) % L::kStages;
          if (n + 1 < nqb &&
              !wait_warp(bar(L::bQFull + st2), ((n + 1) / L::kStages) & 1, abort_flag, p)) {
            ok = false;
            break;
          }
          // S^T(n), dP^T(n) are in registers; P^T(n-1), dS^T(n-1) were
          // written before that.  The gradient products of block n-1 go
          // first: the element-wise warps wait for them before their next
          // P^T store.
          if (!wait_warp(bar(L::bSFree), n & 1, abort_flag, p)) { ok = false; break; }
          ptx::tc_fence_after();
          if (n > 0) issue_g((n - 1) % L::kStages, n > 1);
          if (n + 1 < nqb) issue_s(st2);
        }
        if (ok && wait_warp(bar(L::bPFull), 0, abort_flag, p)) {
          ptx::tc_fence_after();
          issue_g((nqb - 1) % L::kStages, nqb > 1);
        }
      }
      for (int n = 0; !L::kEarly && ok && n < nqb; ++n) {
        const int st = n % L::kStages, st2 = (n + 1) % L::kStages;
        const uint32_t ph2 = ((n + 1) / L::kStages) & 1;
        const bool more = n + 1 < nqb;
        if (L::kEarly && more) {
          if (!wait_warp(bar(L::bQFull + st2), ph2, abort_flag, p) ||
              !wait_warp(bar(L::bSFree), n & 1, abort_flag, p))
            break;
          ptx::tc_fence_after();
          issue_s(st2);
        }
        if (!wait_warp(bar(L::bPFull), n & 1, abort_flag, p)) break;
        ptx::tc_fence_after();
        issue_g(st, n > 0);
        if (!L::kEarly && more) {
          // P^T and dS^T share columns with S^T and dP^T: the next scores go
          // in only after the gradient MMAs (issue order is execution order)
          if (!wait_warp(bar(L::bQFull + st2), ph2, abort_flag, p)) break;
          ptx::tc_fence_after();
          issue_s(st2);
        }
      }
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
    for (int n = 0; n < nqb; ++n) {
      const int i = i_begin + n;
      const int st = n % L::kStages;
      if (!wait_warp(bar(L::bSFull), n & 1, abort_flag, p) ||
          !wait_warp(bar(L::bQFull + st), (n / L::kStages) & 1, abort_flag, p)) {
        ok = false;
        break;
      }
      ptx::tc_fence_after();
      const float *lse_s = reinterpret_cast<const float *>(sm.smem + L::stage(st) + 2 * L::kTile) +
                           h * kBwdHalf;
      const float *d_s = lse_s + kBM;
      // columns (query rows) of this half before `first` do not see the key
      const int first = p.causal ? key - shift - i * kBM - h * kBwdHalf : 0;
      // S^T and dP^T of this half into registers first, so that the next
      // block's products overlap this block's element-wise work
      uint32_t s[kBwdHalf], dp[kBwdHalf];
#pragma unroll
      for (int cc = 0; cc < kBwdHalf; cc += 32) {
        ptx::tmem_ld32(tmem + lane_off + L::tS + h * kBwdHalf + cc,
                       *reinterpret_cast<uint32_t(*)[32]>(&s[cc]));
        ptx::tmem_ld32(tmem + lane_off + L::tdP + h * kBwdHalf + cc,
                       *reinterpret_cast<uint32_t(*)[32]>(&dp[cc]));
      }
      ptx::tmem_wait_ld();
#pragma unroll
      for (int cc = 0; cc < kBwdHalf; cc += 32) {
        ptx::reg_fence32(*reinterpret_cast<uint32_t(*)[32]>(&s[cc]));
        ptx::reg_fence32(*reinterpret_cast<uint32_t(*)[32]>(&dp[cc]));
      }
      ptx::tc_fence_before();
      ptx::mbar_arrive(bar(L::bSFree));
      uint32_t pkp[kBwdHalf / 2], pkd[kBwdHalf / 2];
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
      if (n > 0) {
        // the gradient MMAs of the previous block have read P^T and dS^T
        if (!wait_warp(bar(L::bPDone), (n - 1) & 1, abort_flag, p)) { ok = false; break; }
        ptx::tc_fence_after();
      }
      ptx::tmem_st32(tmem + lane_off + L::tP + h * (kBwdHalf / 2),
                     *reinterpret_cast<uint32_t(*)[32]>(&pkp[0]));
      ptx::tmem_st32(tmem + lane_off + L::tdS + h * (kBwdHalf / 2),
                     *reinterpret_cast<uint32_t(*)[32]>(&pkd[0]));
      ptx::tmem_wait_st();
      ptx::tc_fence_before();
      // (early layout: the MMA thread learns of P^T(n) from the next S-read
      // arrival, so only the last block's is announced here)
      if (!L::kEarly || n == nqb - 1) ptx::mbar_arrive(bar(L::bPFull));
    }
    // ---- epilogue: dV and dK = scale * (dS^T Q), this half's columns
    if (ok && nqb > 0) ok = wait_warp(bar(L::bPDone), (nqb - 1) & 1, abort_flag, p);
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
