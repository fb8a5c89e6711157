/*
 * fa.h -- C ABI of the GB300 (sm_103a) exact attention forward library.
 *
 * The one operation: the exact, IO-aware attention forward pass
 *
 *     O   = softmax(scale * Q K^T [+ causal mask]) V
 *     LSE = per-row natural-log logsumexp of the scaled, masked logits
 *
 * "Scale, mask, softmax and weighted sum" fused into one kernel is how the
 * FlashAttention + TensorRT 10 page describes the fused attention
 * computation (zzycbzc.com/news/393333, section "算子融合的极致优化",
 * item 2).  The IO-aware part -- split the work into blocks that fit in
 * on-chip memory so the N x N matrix never goes to HBM -- is the same
 * page's section "FlashAttention的技术革命", and the "0 MB (recompute)"
 * attention-matrix column of the Flash Attention 2 memory table on the
 * benchmarks page (baguaai.com/zh/skills/benchmarks-332e54, "内存使用分析").
 * The causal flag is the "causal": True setting, required for
 * autoregressive models (2kiu.com/news/1440730, section 3.2).
 *
 * The library computes in fp32 from fp16 or bf16 inputs (mixed precision,
 * 2kiu.com/news/1440730 section 1, item 1) on tcgen05 tensor cores.
 * There is no CPU fallback: every call runs the CUDA kernel or fails.
 */
#ifndef FA_H_
#define FA_H_

#include <stddef.h>

#if defined(__GNUC__)
#define FA_API __attribute__((visibility("default")))
#else
#define FA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* A CUDA stream (cudaStream_t / CUstream); NULL is the legacy default
 * stream. */
struct CUstream_st;
typedef struct CUstream_st *fa_stream_t;

typedef enum {
    FA_OK = 0,
    FA_ERR_NULL = 1,           /* a required pointer is NULL                 */
    FA_ERR_SHAPE = 2,          /* B, H or N negative, or too large           */
    FA_ERR_HEADDIM = 3,        /* d is not 64 or 128                         */
    FA_ERR_DTYPE = 4,          /* dtype is not FA_FP16 or FA_BF16            */
    FA_ERR_ALIGN = 5,          /* q/k/v/o not 16-byte aligned, lse not 4-byte */
    FA_ERR_SCALE = 6,          /* scale is not finite and positive           */
    FA_ERR_CUDA = 7,           /* a CUDA runtime/driver call failed, or the
                                  device is not sm_103 / lacks resources     */
    FA_ERR_DEVICE_TIMEOUT = 8, /* a bounded on-device wait ran out; the
                                  outputs of that launch are undefined      */
    FA_ERR_WORKSPACE = 9       /* workspace missing, misaligned or too small */
} fa_status;

typedef enum { FA_FP16 = 0, FA_BF16 = 1 } fa_dtype;

/*
 * fa_fwd -- attention forward for B*H independent (batch, head) problems.
 *
 *   q, k, v : device pointers, [B, H, N, d] contiguous, element type dtype.
 *   o       : device pointer, [B, H, N, d] contiguous, element type dtype
 *             (written).
 *   lse     : device pointer, [B, H, N] contiguous fp32 (written):
 *             lse[i] = ln(sum over allowed j of exp(scale * q_i . k_j)).
 *   B, H, N : batch, heads, sequence length (queries and keys alike).
 *             Any N >= 1 is accepted; B, H or N equal to 0 is an empty
 *             problem and returns FA_OK without launching anything.
 *   d       : head dimension, 64 or 128.
 *   causal  : nonzero masks key j for query i when j > i.
 *   scale   : multiplier of the logits (usually 1/sqrt(d)); finite and
 *             > 0.
 *   dtype   : FA_FP16 or FA_BF16 (inputs and output alike).
 *   stream  : the CUDA stream the kernel is enqueued on.
 *
 * Ownership: all buffers belong to the caller and must stay valid until
 * the work on `stream` completes.  The library allocates no device memory
 * and keeps no pointer after the call returns.
 *
 * Errors: argument checks happen on the host before anything is enqueued;
 * on any error nothing is launched and the outputs are untouched.  The call
 * is asynchronous: it returns after the launch is enqueued.  Faults on the
 * device (a bounded wait that ran out) are reported by
 * fa_last_device_error().  Pointers to the same buffer for q, k and v are
 * allowed; o and lse must not overlap the inputs or each other.
 */
FA_API fa_status fa_fwd(const void *q, const void *k, const void *v, void *o,
                 float *lse, int B, int H, int N, int d, int causal,
                 float scale, fa_dtype dtype, fa_stream_t stream);

/*
 * fa_fwd_qk -- the same forward pass with different query and key lengths.
 *
 *   q, o    : [B, H, Nq, d];  k, v : [B, H, Nk, d];  lse : [B, H, Nq] fp32.
 *   causal  : key j is visible to query i iff j <= i + (Nk - Nq), i.e. the
 *             mask is aligned to the bottom-right corner (the last query
 *             sees every key; with Nq == Nk this is j <= i).  A query row
 *             that sees no key (i < Nq - Nk) gets O = 0 and LSE = -inf, as
 *             does every row when Nk == 0.
 *   B, H or Nq equal to 0 is an empty problem (FA_OK, nothing launched);
 *   Nk == 0 with Nq > 0 writes the all-masked result.  k and v may be NULL
 *   when Nk == 0.  Everything else as fa_fwd, which equals
 *   fa_fwd_qk(..., Nq = N, Nk = N, ...).
 */
FA_API fa_status fa_fwd_qk(const void *q, const void *k, const void *v,
                           void *o, float *lse, int B, int H, int Nq, int Nk,
                           int d, int causal, float scale, fa_dtype dtype,
                           fa_stream_t stream);

/*
 * fa_fwd_fp8 -- the forward pass on FP8 (e4m3) inputs, with a bf16 output.
 *
 * The FP8 variant is the pages' FlashAttention-3 FP8 column on H100 and
 * its "FP8 precision in commercial use" outlook (baguaai.com benchmarks
 * page, "H100 80GB" table; zzycbzc.com/news/393333, "推理优化的未来方向",
 * item 2).  Both products run on the tcgen05 tensor cores in kind::f8f6f4
 * with fp32 accumulation.
 *
 *   q, k, v : [B, H, Nq|Nk, d] e4m3 (one byte each), 16-byte aligned.  The
 *             real values are q * q_descale, k * k_descale, v * v_descale
 *             (per-tensor descales, finite and > 0).
 *   o       : [B, H, Nq, d] bf16;  lse : [B, H, Nq] fp32 (natural log of the
 *             scaled logits of the real values).
 *   scale, causal, B, H, Nq, Nk, d, stream : as fa_fwd_qk.
 * P (the softmax probabilities, at most 256 under the rescale rule) is
 * rounded to e4m3 for the second product; the row sums use the fp32
 * probabilities.  Errors as fa_fwd_qk, plus FA_ERR_SCALE for a descale that
 * is not finite and positive.
 */
FA_API fa_status fa_fwd_fp8(const void *q, const void *k, const void *v,
                            void *o, float *lse, int B, int H, int Nq, int Nk,
                            int d, int causal, float scale, float q_descale,
                            float k_descale, float v_descale,
                            fa_stream_t stream);

/*
 * fa_fwd_host -- fa_fwd from and to host memory, with the copies overlapped.
 *
 *   q_h, k_h, v_h    : host [B, H, N, d] inputs (page-locked memory lets the
 *                      copies run asynchronously and overlap).
 *   o_h, lse_h       : host outputs, [B, H, N, d] dtype and [B, H, N] fp32.
 *   q_d, k_d, v_d, o_d, lse_d : caller-owned device staging buffers of the
 *                      same shapes (alignment as fa_fwd).
 * The B*H problems are split into chunks; the upload of one chunk, the
 * forward kernel of the previous one and the download of the one before
 * run concurrently on the library's own streams.  All of it is ordered
 * after the work already enqueued on `stream`, and `stream` waits for the
 * last download, so synchronising `stream` makes o_h and lse_h valid.
 * Errors as fa_fwd (checked before anything is enqueued), plus FA_ERR_NULL
 * for a missing host or staging buffer.  A CUDA call that fails part way
 * returns FA_ERR_CUDA; `stream` still waits for every copy and kernel
 * enqueued before the failure, so after synchronising it no copy touches
 * the buffers any more (their contents are then unspecified).
 */
FA_API fa_status fa_fwd_host(const void *q_h, const void *k_h, const void *v_h,
                             void *o_h, float *lse_h, void *q_d, void *k_d,
                             void *v_d, void *o_d, float *lse_d, int B, int H,
                             int N, int d, int causal, float scale,
                             fa_dtype dtype, fa_stream_t stream);

/*
 * fa_bwd_workspace_bytes -- bytes of device workspace fa_bwd needs: two
 * fp32 per query row (scratch derived from the row's logsumexp and from
 * D = rowsum(dout .* o)), each head's N rows rounded up to a multiple of
 * 128: 8 * B * H * ceil(N / 128) * 128 bytes.  0 for an empty problem.
 */
FA_API size_t fa_bwd_workspace_bytes(int B, int H, int N);

/*
 * fa_bwd -- gradients of the attention forward (fa_fwd with the same
 * arguments) for an upstream gradient dout of O.
 *
 *   q, k, v, o, dout : [B, H, N, d] dtype, o and lse as fa_fwd produced them.
 *   lse              : [B, H, N] fp32.
 *   dq, dk, dv       : [B, H, N, d] dtype (written):
 *       dV = P^T dout,  dS = P .* (dout V^T - rowsum(dout .* o)),
 *       dQ = scale * dS K,  dK = scale * dS^T Q,  P = exp(scale Q K^T - lse).
 *   workspace        : caller-owned device memory of at least
 *                      fa_bwd_workspace_bytes(B, H, N) bytes, 16-byte
 *                      aligned; its contents on entry do not matter, and
 *                      calls that run concurrently need separate workspaces.
 * P is recomputed from q, k and lse, never stored: the attention matrix
 * costs no memory in the backward either ("0 MB (recompute)" in the Flash
 * Attention 2 memory table, baguaai.com/zh/skills/benchmarks-332e54,
 * "内存使用分析"; the same page lists training performance, i.e. forward
 * and backward, among its benchmarks).  The gradient formulas are the
 * chain rule through softmax(scale Q K^T) V.  Three kernels are
 * enqueued on `stream` (row sums, dQ, then dK and dV).  Errors as fa_fwd,
 * plus FA_ERR_WORKSPACE.  d is 64 or 128; dtype FA_FP16 or FA_BF16.
 */
FA_API fa_status fa_bwd(const void *q, const void *k, const void *v,
                        const void *o, const void *dout, const float *lse,
                        void *dq, void *dk, void *dv, void *workspace,
                        size_t workspace_bytes, int B, int H, int N, int d,
                        int causal, float scale, fa_dtype dtype,
                        fa_stream_t stream);

/*
 * fa_bwd_noalloc -- fa_bwd for callers that cannot allocate device memory.
 *
 * The pages have no counterpart of this entry point.  It exists for code
 * that must not call cudaMalloc or an allocator of its own: for instance a
 * plug-in running inside a host program that owns every device allocation,
 * or a latency-bound loop that may not pay for an allocation.  fa_bwd needs
 * a workspace of fa_bwd_workspace_bytes(B, H, N) bytes; this variant uses a
 * fixed array in the library's static device memory instead, so it takes no
 * workspace argument and allocates nothing.
 *
 * Limit: B * H * ceil(N / 128) * 128 <= FA_BWD_NOALLOC_MAX_ROWS (2^21;
 * two fp32 per row: 16 MiB held on every device that loads the library,
 * until the process exits).  Larger problems return FA_ERR_WORKSPACE
 * without touching the device; use fa_bwd with a workspace for them.
 *
 * The first call on a device looks up the array's device address (once per
 * device, with that device current); make that first call before any stream
 * capture.  Every call shares the one array and leaves its contents behind;
 * each call fully rewrites the part it reads, so nothing needs clearing, but
 * calls that overlap on the GPU (different streams, or different host
 * threads on one device) race on it and must be ordered by the caller.
 * Arguments, results and other errors are those of fa_bwd.
 */
#define FA_BWD_NOALLOC_MAX_ROWS (1LL << 21)
FA_API fa_status fa_bwd_noalloc(const void *q, const void *k, const void *v,
                                const void *o, const void *dout,
                                const float *lse, void *dq, void *dk, void *dv,
                                int B, int H, int N, int d, int causal,
                                float scale, fa_dtype dtype,
                                fa_stream_t stream);

/* A static, human-readable description of a status code. */
FA_API const char *fa_status_string(fa_status status);

/*
 * fa_last_device_error -- synchronise `stream`, then report and clear the
 * device-side status word of the current device.
 *
 * Every wait inside the kernel is bounded in time; a wait that runs out
 * records a flag in a per-device status word and the kernel returns
 * early (its TMEM released).  This call returns FA_ERR_DEVICE_TIMEOUT if
 * any launch since the previous call recorded such a flag, FA_ERR_CUDA if
 * the synchronisation itself failed, and FA_OK otherwise.
 */
FA_API fa_status fa_last_device_error(fa_stream_t stream);

/* The library's version as major * 10000 + minor * 100 + patch. */
FA_API int fa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FA_H_ */
