/*
 * C ABI of the GB300 (sm_103a) tiled online-softmax attention library.
 *
 * Tensors are plain device pointers; sizes are ints; nothing here depends on
 * a framework.  Every call is asynchronous on the given CUDA stream (passed as
 * `void*`, i.e. a cudaStream_t; NULL = the legacy default stream).  Argument
 * errors are reported synchronously by the return value and launch nothing.
 * The caller allocates and owns every buffer, including the backward
 * workspace; the library keeps only a per-device SM-count cache.
 *
 * Layouts (all contiguous, row-major):
 *   Q, O, dO, dQ   [B, L, H,   D]   fp16 or bf16 ("BSHD")
 *   K, V, dK, dV   [B, L, Hkv, D]   same dtype as Q
 *   LSE, Delta     [B, H, L]        fp32
 * Query head h reads K/V head h / (H / Hkv) (grouped-query attention).
 * The softmax scale is fixed at 1 / sqrt(D).  Causal masking is top-left
 * aligned with one length L for queries and keys: key j is visible to query i
 * iff j <= i.  Every pointer must be 16-byte aligned.
 * Supported: D in {64, 128}; L >= 1; B, H, Hkv >= 1 with H % Hkv == 0;
 * B * H * L and B * L * H * D must fit the kernels' 32-bit coordinates
 * (B, L, H < 2^31 and B * L * H * D < 2^40).
 */
#ifndef TILED_ATTENTION_FA_GB300_FA_H
#define TILED_ATTENTION_FA_GB300_FA_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  FA_OK = 0,
  FA_ERR_INVALID_ARG = 1,    /* null/misaligned pointer, bad size, H % Hkv != 0 */
  FA_ERR_UNSUPPORTED = 2,    /* D or dtype outside the supported set, or the device or the
                                build cannot run the kernel as designed (too little shared
                                memory per block; a backward kernel compiled with a register
                                allocation other than its warpgroup split assumes);
                                nothing was launched */
  FA_ERR_CUDA = 3,           /* a CUDA runtime call or kernel launch failed */
  FA_ERR_DEVICE_TIMEOUT = 4, /* a kernel gave up a bounded wait (see fa_check_device_error) */
  FA_ERR_SCRATCH_TOO_SMALL = 5 /* fa_bwd_noalloc's fixed scratch or fa_decode's workspace is
                                  smaller than the problem needs; nothing was launched */
} fa_status;

typedef enum { FA_F16 = 0, FA_BF16 = 1 } fa_dtype;

/*
 * Forward attention.  For each batch b and query head h:
 *   S = Q_bh K_bh'^T / sqrt(D)   (h' = h / (H / Hkv)), causal: S_ij = -inf for j > i
 *   O_bh = softmax_rows(S) V_bh'                 -> O   [B, L, H, D]
 *   LSE_bh,i = ln sum_j exp(S_ij)                -> LSE [B, H, L], fp32
 * Page "使用 TileLang 在 AMD GPU 上快速开发高性能 Flash Attention", sections
 * 核心公式与计算流程 (the formulas) and K/V Tile 遍历与核心计算 (the tiled
 * online-softmax loop this kernel implements); the LSE is the per-row
 * statistic the backward kernel of page "TileLang与机器学习训练：反向传播算子优化案例"
 * takes as input (section 算子拆分与流水线设计).
 * Q, K, V are read only.  O and LSE are written in full (LSE may not be NULL).
 */
fa_status fa_fwd(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int L,
                 int H, int Hkv, int D, int causal, int dtype, void* stream);

/*
 * Forward with fewer queries than keys (prefill against a key/value cache):
 * Q, O [B, Lq, H, D]; K, V [B, Lk, Hkv, D]; LSE [B, H, Lq].  Under causal
 * masking the queries are the last Lq positions of the Lk-long sequence:
 * query i sees key j iff j <= i + past_len with past_len = Lk - Lq (page
 * "TileLang性能分析报告：H100上FlashAttention吞吐量达1.2PFlops", section
 * 因果掩码优化, where the query index is the row plus past_len); causal
 * calls need Lk >= Lq.  Non-causal calls accept any Lq, Lk >= 1.  With
 * Lq == Lk this is fa_fwd.
 */
fa_status fa_fwd_kv(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int Lq,
                    int Lk, int H, int Hkv, int D, int causal, int dtype, void* stream);

/*
 * Forward on 8-bit inputs: Q8, K8, V8 hold E4M3 codes (one byte per element,
 * the OCP 8-bit floating point E4M3 format without infinities), in the
 * layouts above, each with one fp32 scale: the call computes the fa_fwd_kv
 * result (same masking rule, past_len = Lk - Lq) for the dequantised inputs
 *   Q = decode(Q8) * q_scale,  K = decode(K8) * k_scale,  V = decode(V8) * v_scale,
 * writing O [B, Lq, H, D] in `out_dtype` (FA_F16 or FA_BF16) and LSE
 * [B, H, Lq] in fp32.  Page "TileLang性能分析报告：H100上FlashAttention吞吐量达
 * 1.2PFlops", section 生产环境部署建议, item 1 (FP8 mixed-precision compute);
 * the loop is the online softmax of page "使用 TileLang 在 AMD GPU 上快速开发
 * 高性能 Flash Attention", section K/V Tile 遍历与核心计算, with P rounded to
 * E4M3 before the PV product, as that page rounds P to the input type.
 * Scores accumulate in fp32 from exact products; the rounding of P is the
 * one approximation (relative error at most 2^-4 per probability, absolute
 * 2^-10 below 2^-6).  Requires D = 128 (FA_ERR_UNSUPPORTED otherwise) and
 * finite scales > 0 (FA_ERR_INVALID_ARG otherwise).
 */
fa_status fa_fwd_fp8(const void* Q8, const void* K8, const void* V8, float q_scale,
                     float k_scale, float v_scale, void* O, float* LSE, int B, int Lq, int Lk,
                     int H, int Hkv, int D, int causal, int out_dtype, void* stream);

/*
 * Split-KV decoding: the forward of fa_fwd_kv (same result, layouts, masking
 * rule and causal past_len = Lk - Lq) computed for few queries against many
 * keys.  The keys of each (batch, K/V head) are cut into equal slices of
 * 128-key tiles, one CTA per slice, sized so the slices fill the GPU; each
 * slice yields a partial output and log-sum-exp in fp32, and a second kernel
 * merges them: LSE = ln sum_s exp(LSE_s), O = sum_s exp(LSE_s - LSE) O_s.
 * Page "TileLang性能分析报告：H100上FlashAttention吞吐量达1.2PFlops", section
 * 生产环境部署建议 (item 2 names flash_decoding for inference; the slicing and
 * merge are the plain reading of that name); the per-slice loop is the online
 * softmax of page "使用 TileLang 在 AMD GPU 上快速开发高性能 Flash Attention",
 * section K/V Tile 遍历与核心计算.
 * The g = H / Hkv query heads of a K/V head and all Lq queries share one
 * 128-row tile, so the call requires g * Lq <= 128 (FA_ERR_UNSUPPORTED
 * otherwise; use fa_fwd_kv).  `workspace` is the caller's device buffer of
 * `workspace_bytes` (16-byte aligned) holding the partials; it needs
 * fa_decode_workspace_size(...) bytes, asked with the same sizes and with the
 * device that will run the call current (the slice count depends on its SM
 * count).  Smaller buffers return FA_ERR_SCRATCH_TOO_SMALL and launch nothing.
 * Its contents need no initialisation and are unspecified afterwards; calls
 * that overlap on the GPU must not share one workspace.
 */
size_t fa_decode_workspace_size(int B, int Lq, int Lk, int H, int Hkv, int D);
fa_status fa_decode(const void* Q, const void* K, const void* V, void* O, float* LSE,
                    void* workspace, size_t workspace_bytes, int B, int Lq, int Lk, int H, int Hkv,
                    int D, int causal, int dtype, void* stream);

/*
 * The two stages fa_decode runs, for callers that schedule or time them
 * apart: fa_decode_slices writes every slice's partial O and LSE into the
 * workspace; fa_decode_merge reads them and writes O and LSE.  Give both the
 * same sizes and run them on the same device, so that they derive the same
 * slice plan; the merge must run after the slices on the stream.
 */
fa_status fa_decode_slices(const void* Q, const void* K, const void* V, void* workspace,
                           size_t workspace_bytes, int B, int Lq, int Lk, int H, int Hkv, int D,
                           int causal, int dtype, void* stream);
fa_status fa_decode_merge(const void* workspace, size_t workspace_bytes, void* O, float* LSE, int B,
                          int Lq, int Lk, int H, int Hkv, int D, int dtype, void* stream);

/*
 * Backward preprocess: Delta[b, h, i] = sum_d O[b, i, h, d] * dO[b, i, h, d]
 * (fp32 accumulation), the per-row term of the softmax gradient.  Page
 * "TileLang与机器学习训练：反向传播算子优化案例", section 算子拆分与流水线设计
 * (the "Delta" preprocessing stage; its printed block product is read as this
 * per-row dot product).  When `dq_accum` is not NULL it must point to
 * fa_bwd_workspace_size(B, L, H, D) bytes, which this call sets to zero in
 * the same pass, ready for fa_bwd.
 */
fa_status fa_bwd_preprocess(const void* O, const void* dO, float* Delta, float* dq_accum, int B,
                            int L, int H, int D, int dtype, void* stream);

/* Bytes of the fp32 dQ accumulator fa_bwd needs: B * H * ceil(L/128)*128 * D * 4. */
size_t fa_bwd_workspace_size(int B, int L, int H, int D);

/*
 * Backward attention: dQ, dK, dV of the forward above, given dO, the forward's
 * LSE and fa_bwd_preprocess's Delta.  With P = exp(S - LSE):
 *   dV = P^T dO,  dP = dO V^T,  dS = P o (dP - Delta),
 *   dQ = dS K / sqrt(D),  dK = dS^T Q / sqrt(D),
 * with dK, dV of a K/V head summed over its query heads.  Page
 * "TileLang与机器学习训练：反向传播算子优化案例", sections 算子拆分与流水线设计
 * (one K/V tile per CTA looping over Q tiles, dV accumulated from the
 * transposed probabilities) and 内存布局优化 (dQ accumulated in fp32 through
 * atomics into a layout matched to the accumulator fragments, then a
 * post-processing pass).
 * `dq_accum` is the caller's workspace (fa_bwd_workspace_size bytes, 16-byte
 * aligned); it must hold zeros on entry unless `zero_accum` is non-zero, in
 * which case this call zeroes it first.  Its contents afterwards are
 * unspecified.  O is accepted for interface symmetry and is not read (Delta
 * carries it); it may be NULL.  dQ, dK, dV are written in full.
 */
fa_status fa_bwd(const void* Q, const void* K, const void* V, const void* O, const void* dO,
                 const float* LSE, const float* Delta, void* dQ, void* dK, void* dV,
                 float* dq_accum, int zero_accum, int B, int L, int H, int Hkv, int D, int causal,
                 int dtype, void* stream);

/*
 * Backward of fa_fwd_kv: Q, O, dO, dQ [B, Lq, H, D]; K, V, dK, dV
 * [B, Lk, Hkv, D]; LSE, Delta [B, H, Lq]; dq_accum of
 * fa_bwd_workspace_size(B, Lq, H, D) bytes (fa_bwd_preprocess with L = Lq
 * computes Delta and zeroes it).  Same masking rule and limits as fa_fwd_kv.
 */
fa_status fa_bwd_kv(const void* Q, const void* K, const void* V, const void* O, const void* dO,
                    const float* LSE, const float* Delta, void* dQ, void* dK, void* dV,
                    float* dq_accum, int zero_accum, int B, int Lq, int Lk, int H, int Hkv, int D,
                    int causal, int dtype, void* stream);

/*
 * The two stages fa_bwd runs, for callers that schedule or time them apart:
 *   fa_bwd_main        dK, dV (written in full) and the dQ accumulator (added
 *                      into; it must hold zeros on entry unless zero_accum);
 *   fa_bwd_postprocess dQ = dq_accum / sqrt(D), converted back to BSHD.
 * Page "TileLang与机器学习训练：反向传播算子优化案例", section
 * 算子拆分与流水线设计 (the core gradient stage and the post-processing stage
 * that reorders the dQ gradient).  Arguments mean what they mean for fa_bwd.
 */
fa_status fa_bwd_main(const void* Q, const void* K, const void* V, const void* dO,
                      const float* LSE, const float* Delta, void* dK, void* dV, float* dq_accum,
                      int zero_accum, int B, int L, int H, int Hkv, int D, int causal, int dtype,
                      void* stream);
fa_status fa_bwd_postprocess(const float* dq_accum, void* dQ, int B, int L, int H, int D,
                             int dtype, void* stream);

/*
 * fa_bwd for callers that cannot allocate device memory at call time: a
 * plugin running inside a host application that owns all GPU memory through
 * its own pool and hands out no allocator, or a serving path that must not
 * allocate once it has started.  This is a library facility; the pages have
 * no counterpart.
 * Same arguments and results as fa_bwd, minus the workspace.  Such a caller
 * gets Delta from fa_bwd_preprocess with a NULL dq_accum (which needs no
 * workspace either).  The fp32 dQ
 * accumulator lives in a fixed device array of FA_NOALLOC_SCRATCH_BYTES that
 * the library's module holds on every GPU that loads it, until exit.  The
 * call allocates nothing (no cudaMalloc, cudaFree or allocating library
 * routine); it clears the part of the array it uses, then runs the backward.
 * Limits and rules:
 *   - B * H * ceil(L/128)*128 * D * 4 bytes must not exceed
 *     FA_NOALLOC_SCRATCH_BYTES (64 MiB, e.g. B=1, H=32, L=4096, D=128);
 *     larger problems return FA_ERR_SCRATCH_TOO_SMALL and launch nothing.
 *   - Every call on a device shares the one array: calls whose work overlaps
 *     on the GPU (other streams, other host threads) race and corrupt each
 *     other's dQ.  Serialise them.
 *   - Each call looks up the array's device address on the current device
 *     (the address can change if the device is reset and the module loaded
 *     again) and remembers it; a call made while its stream is being
 *     captured uses the remembered address instead.  Make the first call on
 *     each device before any stream capture on that device.
 */
#define FA_NOALLOC_SCRATCH_BYTES ((size_t)64 << 20)
fa_status fa_bwd_noalloc(const void* Q, const void* K, const void* V, const void* O,
                         const void* dO, const float* LSE, const float* Delta, void* dQ,
                         void* dK, void* dV, int B, int L, int H, int Hkv, int D, int causal,
                         int dtype, void* stream);

/*
 * Synchronise `stream` and report whether any kernel of this library gave up
 * a bounded wait since the last check (FA_ERR_DEVICE_TIMEOUT; the word is then
 * cleared).  Kernels never trap or spin forever: a wait that exceeds about one
 * second records its site id, unwinds the CTA and returns.
 */
fa_status fa_check_device_error(void* stream);

/*
 * Exercise the bounded-wait failure path without any fault: launches one
 * thread that waits on an mbarrier nothing ever completes.  After
 * `limit_ns` (clamped to 1 ms .. 1 s) the wait gives up, records site 900 in
 * the device error word and the kernel returns; the next
 * fa_check_device_error on the stream then returns FA_ERR_DEVICE_TIMEOUT and
 * the CUDA context stays usable.  A library facility with no counterpart on
 * the pages.
 */
fa_status fa_selftest_bounded_wait(unsigned long long limit_ns, void* stream);

/* Site id recorded by the last FA_ERR_DEVICE_TIMEOUT (0 if none). */
unsigned int fa_last_error_site(void);

/* Static, human-readable text for a status value. */
const char* fa_status_string(fa_status status);

/* Library version string. */
const char* fa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* TILED_ATTENTION_FA_GB300_FA_H */
