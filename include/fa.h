/*
 * fa.h -- C ABI of the GB300 (sm_103a) exact tiled attention forward.
 *
 * One call computes, for every batch b, query head h and query row i,
 *
 *   o[b,h,i,:] = sum_{j in V_i} e^{s_ij} v_j / ( sum_{j in V_i} e^{s_ij} + e^{z_h} )
 *   lse[b,h,i] = log( sum_{j in V_i} e^{s_ij} + e^{z_h} )
 *   s_ij       = scale * q_i . k_j + mask[b,h,i,j]
 *   V_i        = { j < Tk : (causal == 0 or j <= p_i) and (window <= 0 or j > p_i - window) }
 *   p_i        = q_offset + i
 *
 * as defined on "FlashAttention forward in C" (section 2.1, "What is
 * computed", and section 4, "The interface") with the strided additive mask of
 * "Fused attention and softmax: fast and exact" ("What is computed").  The
 * e^{z_h} term is present only when sinks are given.  Query head h reads KV
 * head floor(h / (Hq / Hkv)).  A row with no visible key (after the mask) and
 * no sink gives o = 0 and lse = -inf; with a sink it gives o = 0 and lse = z_h.
 * The [Tq, Tk] score matrix is never stored: keys are walked one tile at a
 * time under an online softmax ("FlashAttention forward in C", section 2.2).
 *
 * Layout (all tensors contiguous, row-major, element strides implied):
 *   q, o   [B, Hq,  Tq, d]   in `dtype`
 *   k, v   [B, Hkv, Tk, d]   in `dtype`
 *   lse    [B, Hq,  Tq]      float32, or NULL to skip it
 *   sinks  [Hq]              float32 raw logits (not scaled, not masked), or NULL
 *   mask   float32, element (b,h,i,j) at mask[b*mask_sb + h*mask_sh + i*mask_sq + j*mask_sk];
 *          strides in elements, >= 0, a stride of 0 broadcasts; NULL for no mask.
 *          Entries may be finite or -inf; +inf and NaN are outside the domain.
 * All pointers are DEVICE pointers on the current CUDA device.  q, k, v and o
 * must be 16-byte aligned.  The caller owns every buffer; the library keeps
 * no state between calls beyond cached kernel attributes and allocates no
 * device memory.  The attributes are set by the first call of the process on
 * the device then current: a process drives one GPU, and its first call is
 * not made from several host threads at once.
 *
 * Arithmetic: FA_DTYPE_F32 computes in fp32 on the SIMT cores (FFMA) and
 * writes fp32 o.  FA_DTYPE_BF16 reads bf16 q/k/v, forms S = Q K^T and O = P V
 * on the tcgen05 tensor cores with fp32 accumulators in tensor memory, keeps
 * the softmax statistics in fp32, rounds P to bf16 for the P.V product, and
 * writes bf16 o (round to nearest even).  FA_DTYPE_F32_TC reads and writes
 * fp32 like FA_DTYPE_F32 but forms both products on the tcgen05 tensor cores,
 * three products per matrix product with fp32 accumulation: S = Q K^T in TF32
 * mode as Q_hi K_hi + Q_hi K_lo + Q_lo K_hi, where x_hi is x with its low 13
 * mantissa bits cleared (the part TF32 keeps) and x_lo = x - x_hi (a logit's
 * error ~2^-20 of sum |q_i k_i|); O = P V in bf16 as P_0 V_0 + P_0 V_1 +
 * P_1 V_0 with x_0 = bf16(x), x_1 = bf16(x - x_0) (~2^-17 of sum |p_j v_j|).
 * FA_DTYPE_FP8_E4M3 reads e4m3 q/k/v (OCP FP8 E4M3, one byte each: the
 * layout rows above in bytes), forms S = Q K^T and O = P V on the tensor cores
 * (kind::f8f6f4, fp32 accumulators), keeps the softmax statistics in fp32,
 * rounds P to e4m3 for the P.V product, and writes bf16 o.  Scaling of the
 * inputs into e4m3's range is the caller's: a per-tensor descale of q and k
 * folds into `scale`, and o is linear in v.  lse is fp32 in all four.
 *
 * Execution: asynchronous on `stream` (a cudaStream_t, NULL = legacy default
 * stream); results are valid once the stream has synchronised.
 *
 * Errors are reported before any launch and before anything is written:
 *   FA_EINVAL        negative sizes or q_offset, a NULL q/o when B*Hq*Tq > 0,
 *                    a NULL k/v when Tk > 0 (and B*Hq*Tq > 0), an unknown
 *                    dtype, a non-finite scale, a negative mask stride, sizes
 *                    whose element counts overflow.
 *   FA_ESHAPE        Hq % Hkv != 0, Hkv > Hq, or Hkv == 0 with Hq > 0
 *                    ("FlashAttention forward in C", section 4: TL_ESHAPE).
 *   FA_EUNSUPPORTED  d odd or 0 ("Fused attention and softmax": d must be
 *                    even), d > 256 for fp32, bf16 d not a multiple of 8
 *                    or above 128 (rows must be 16-byte multiples for TMA),
 *                    FA_DTYPE_F32_TC d not a multiple of 4 or above 128,
 *                    FA_DTYPE_FP8_E4M3 d not a multiple of 16 or above 128,
 *                    B*Hq*ceil(Tq/128) >= 2^31 on the tensor-core dtypes
 *                    (bf16, F32_TC, e4m3), B*Hq*ceil(Tq/64) >= 2^31 for
 *                    FA_DTYPE_F32, Tq or Tk >= 2^30, pointers not 16-byte
 *                    aligned.
 *   FA_ECUDA         a CUDA error while configuring or launching.
 * B*Hq*Tq == 0 is a no-op returning FA_OK.  Tk == 0 writes o = 0 and
 * lse = -inf (or the sink).  fa_last_error() describes the last non-OK
 * status returned on the calling thread.
 */
#ifndef FA_GB300_FA_H
#define FA_GB300_FA_H

#include <stdint.h>
#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    FA_OK = 0,
    FA_EINVAL = 1,
    FA_ESHAPE = 2,
    FA_EUNSUPPORTED = 3,
    FA_ECUDA = 4,
    FA_ETIMEOUT = 5
} fa_status;

typedef enum {
    FA_DTYPE_F32 = 0,
    FA_DTYPE_BF16 = 1,
    FA_DTYPE_F32_TC = 2,
    FA_DTYPE_FP8_E4M3 = 3
} fa_dtype;

/* The attention forward described above.  `dtype` is an fa_dtype value;
 * `stream` is a cudaStream_t passed as void* so that this header needs no
 * CUDA include. */
fa_status fa_fwd(const void *q, const void *k, const void *v, void *o, float *lse,
                 int64_t B, int64_t Hq, int64_t Hkv, int64_t Tq, int64_t Tk, int64_t d,
                 float scale, int64_t q_offset, int causal, int64_t window,
                 const float *sinks,
                 const float *mask, int64_t mask_sb, int64_t mask_sh, int64_t mask_sq, int64_t mask_sk,
                 int dtype, void *stream);

/* The same computation on strided tensors (the layouts of engines that keep
 * [B, T, H, d] or [T, H*d] buffers; "FlashAttention forward in C" works on
 * [B, H, T, d] only).  Element (b, h, t, x) of q is at
 * q[b*q_sb + h*q_sh + t*q_st + x], likewise k, v (with Hkv, Tk) and o; the d
 * elements of a row are contiguous.  lse stays contiguous [B, Hq, Tq].
 * fa_fwd(...) is this call with q_sb = Hq*Tq*d, q_sh = Tq*d, q_st = d (and so
 * on).  Additional errors:
 *   FA_EINVAL        a negative stride of a dimension of extent > 1, an
 *                    extent overflowing int64, or o strides that make two
 *                    output rows overlap (checked by the rule "every stride,
 *                    in increasing order, covers the span of the smaller
 *                    dimensions").
 *   FA_EUNSUPPORTED  bf16: a stride (of a dimension of extent > 1) that is
 *                    not a multiple of 8 elements (16 bytes, a TMA rule) or
 *                    reaches 2^40 bytes; FA_DTYPE_F32_TC: likewise with 4
 *                    elements; FA_DTYPE_FP8_E4M3: 16 elements for q, k, v
 *                    and 8 for the bf16 o; fp32: a stride that is odd.
 * Reading k or v through overlapping rows (a stride of 0 over the batch, say)
 * is allowed for FA_DTYPE_F32; the tensor-core paths need positive strides. */
fa_status fa_fwd_strided(const void *q, const void *k, const void *v, void *o, float *lse,
                         int64_t B, int64_t Hq, int64_t Hkv, int64_t Tq, int64_t Tk, int64_t d,
                         int64_t q_sb, int64_t q_sh, int64_t q_st,
                         int64_t k_sb, int64_t k_sh, int64_t k_st,
                         int64_t v_sb, int64_t v_sh, int64_t v_st,
                         int64_t o_sb, int64_t o_sh, int64_t o_st,
                         float scale, int64_t q_offset, int causal, int64_t window,
                         const float *sinks,
                         const float *mask, int64_t mask_sb, int64_t mask_sh, int64_t mask_sq, int64_t mask_sk,
                         int dtype, void *stream);

/* Decode steps against paged K/V caches (the consumer named on "FlashAttention
 * forward in C", section 5: paged attention performs the same tile update on
 * blocks and is held to this kernel bit for bit).  Sequence b holds
 * seq_lens[b] keys (device int32 [B], at most max_seq_len); its Tq queries
 * q[b, :, 0..Tq) are its last Tq positions (q_offset_b = seq_lens[b] - Tq,
 * the rows below 0 seeing no key).  Key j of sequence b and KV head g is
 * k_cache[page, j % page_size, g, :] with page = block_table[b * max_blocks +
 * j / page_size] (device int32); the caches are contiguous
 * [num_pages, page_size, Hkv, d], q and o contiguous [B, Hq, Tq, d], lse
 * [B, Hq, Tq].  Page indices outside [0, num_pages) read as zero keys; table
 * entries past a sequence's keys are never read.  The flags are those of
 * fa_fwd (no additive mask).  Errors as fa_fwd, plus:
 *   FA_EINVAL        max_seq_len > max_blocks * page_size; NULL seq_lens, or
 *                    NULL caches / block_table with max_seq_len > 0.
 *   FA_EUNSUPPORTED  dtype other than bf16; (Hq / Hkv) * Tq > 128;
 *                    page_size neither a divisor of 128 (>= 8) nor a multiple
 *                    of 128; num_pages, max_blocks or page_size >= 2^31.
 * A sequence's result equals that of fa_fwd on its keys laid out
 * contiguously, bit for bit, when both calls split the key range the same
 * way (same B, Hkv and longest length). */
fa_status fa_fwd_paged(const void *q, const void *k_cache, const void *v_cache, void *o, float *lse,
                       int64_t B, int64_t Hq, int64_t Hkv, int64_t Tq, int64_t d,
                       const int32_t *seq_lens, int64_t max_seq_len,
                       const int32_t *block_table, int64_t max_blocks,
                       int64_t page_size, int64_t num_pages,
                       float scale, int causal, int64_t window, const float *sinks,
                       int dtype, void *stream);

/* Split-KV decode through a caller-owned workspace (Flash-Decoding, named on
 * "FlashAttention forward in C", section 5, beside the fixed tile order: long
 * contexts are split across thread blocks and the partial (m, l, a) merged
 * with the same rescale, which trades invariance for parallelism).  Same
 * arguments, layout and result as fa_fwd.  When every query row of a KV group
 * fits one 128-row tile ((Hq / Hkv) * Tq <= 128) and dtype is bf16, each
 * (batch, KV head) is split over S CTAs (S = SM count / (B * Hkv), 1..64, at
 * least two key tiles each), not over one thread-block cluster as fa_fwd
 * does: every SM gets work however few KV heads there are.  Each CTA writes
 * its unnormalised fp32 O and (m, l) per row into the workspace; the last CTA
 * of a KV head to finish merges them, in split order, into o and lse.  Other
 * calls (other dtypes, larger groups) run exactly as fa_fwd and ignore the
 * workspace.
 *   workspace        device memory of at least the size that
 *                    fa_splitkv_workspace_bytes reports for these sizes,
 *                    16-byte aligned, owned by the caller; its contents
 *                    before and after the call are scratch.  A call clears
 *                    the counters it uses (a memset on `stream`) before its
 *                    kernel, so the same workspace serves any number of
 *                    calls in stream order; calls that run at the same time
 *                    need separate workspaces.
 * The split count depends on B * Hkv and the SM count, so results agree with
 * fa_fwd within rounding, not bit for bit, and are not batch-invariant.
 * Errors as fa_fwd, plus FA_EINVAL for a NULL, short or unaligned workspace
 * when the call needs one. */
fa_status fa_fwd_splitkv(const void *q, const void *k, const void *v, void *o, float *lse,
                         int64_t B, int64_t Hq, int64_t Hkv, int64_t Tq, int64_t Tk, int64_t d,
                         float scale, int64_t q_offset, int causal, int64_t window,
                         const float *sinks,
                         const float *mask, int64_t mask_sb, int64_t mask_sh, int64_t mask_sq, int64_t mask_sk,
                         void *workspace, size_t workspace_bytes, int dtype, void *stream);

/* The workspace size in bytes that fa_fwd_splitkv needs for these sizes on
 * the current device (0 when the call takes another path).  Host-only; it
 * reads the device's SM count once.  FA_EINVAL for NULL `bytes`, an unknown
 * dtype or a negative size; FA_ESHAPE when Hq is not a multiple of Hkv. */
fa_status fa_splitkv_workspace_bytes(int64_t B, int64_t Hq, int64_t Hkv, int64_t Tq, int64_t d, int dtype,
                                     size_t *bytes);

/* Size in bytes of the device array that fa_fwd_splitkv_noalloc uses as its
 * workspace: 4 MiB, held by every GPU that loads this library until the
 * process exits. */
#define FA_SPLITKV_NOALLOC_MAX_SCRATCH ((size_t)4 << 20)

/* fa_fwd_splitkv for callers that must not allocate device memory.  This
 * entry point is a service of the library; the paper has no counterpart.
 * Some callers cannot call cudaMalloc or hand out a buffer of their own:
 *   - an inference engine whose memory planner has already reserved the GPU's
 *     memory and accounts for every byte;
 *   - a plugin whose host forbids allocation inside its execute callback;
 *   - a latency-critical loop where cudaMalloc, which can synchronise the
 *     device, would stall the pipeline.
 * They still pass q, k, v, o and lse, with the arguments and layout of fa_fwd.
 * The split-KV workspace is a static device array of
 * FA_SPLITKV_NOALLOC_MAX_SCRATCH bytes inside the library.  Neither this call
 * nor anything it reaches calls cudaMalloc, cudaFree or an allocating library
 * routine.
 *   - Size limit: a call whose workspace (fa_splitkv_workspace_bytes) exceeds
 *     the array fails with FA_EUNSUPPORTED and a message giving both sizes.
 *     Nothing is launched.  Use fa_fwd_splitkv with a workspace of that size
 *     instead.  Calls that need no workspace run exactly as fa_fwd.
 *   - First call on a device: it looks up the array's device address on the
 *     current device, once per device.  Make that first call before any
 *     stream capture.
 *   - Sharing: every call on a device shares the one array, and the array
 *     keeps whatever the previous call left in it.  Each call clears the
 *     counters it needs (a memset on `stream`) before its kernel.  Calls in
 *     stream order are safe.  Calls whose work overlaps on the GPU race on the
 *     array and give wrong results: other streams, or other host threads on
 *     the same device.
 * Results, invariance and other errors are those of fa_fwd_splitkv. */
fa_status fa_fwd_splitkv_noalloc(const void *q, const void *k, const void *v, void *o, float *lse,
                                 int64_t B, int64_t Hq, int64_t Hkv, int64_t Tq, int64_t Tk, int64_t d,
                                 float scale, int64_t q_offset, int causal, int64_t window,
                                 const float *sinks,
                                 const float *mask, int64_t mask_sb, int64_t mask_sh, int64_t mask_sq,
                                 int64_t mask_sk, int dtype, void *stream);

/* A variable-length batch: B sequences packed along the rows of q, o
 * ([total_q, Hq, d]) and k, v ([total_k, Hkv, d]), element (t, h, x) of q at
 * q[h*q_sh + t*q_st + x] (likewise k, v, o), d contiguous.  Sequence b has the
 * rows [cu_seqlens_q[b], cu_seqlens_q[b+1]) of q and o and [cu_seqlens_k[b],
 * cu_seqlens_k[b+1]) of k and v (device int32 [B+1], non-decreasing); its
 * queries are its last positions (q_offset_b = its keys - its queries), which
 * makes Tq = Tk a causal prefill and fewer queries a chunk or a decode step.
 * lse is contiguous [Hq, total_q].  max_seqlen_q bounds every sequence's
 * query count (it sizes the grid; rows past it are not computed);
 * max_seqlen_k is the analogous bound on keys.  Offsets are clamped into
 * [0, total], so a malformed table cannot make the kernels reach outside the
 * tensors.  No additive mask.  Errors as fa_fwd_strided, plus FA_EINVAL for a
 * NULL cu_seqlens table and FA_EUNSUPPORTED when max_seqlen_q > total_q,
 * B*Hq*ceil(max_seqlen_q/128) >= 2^31 (64 for FA_DTYPE_F32), or dtype is
 * FA_DTYPE_F32_TC (fp32 batches run on FA_DTYPE_F32 here).  With
 * FA_DTYPE_FP8_E4M3, q, k and v are e4m3 (strides multiples of 16 elements)
 * and o is bf16 (strides multiples of 8). */
fa_status fa_fwd_varlen(const void *q, const void *k, const void *v, void *o, float *lse,
                        int64_t B, int64_t Hq, int64_t Hkv, int64_t d,
                        const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k,
                        int64_t total_q, int64_t total_k, int64_t max_seqlen_q, int64_t max_seqlen_k,
                        int64_t q_sh, int64_t q_st, int64_t k_sh, int64_t k_st,
                        int64_t v_sh, int64_t v_st, int64_t o_sh, int64_t o_st,
                        float scale, int causal, int64_t window, const float *sinks,
                        int dtype, void *stream);

/* Message for the last non-OK status on this thread ("" if none).  The
 * pointer stays valid until the next fa_* call on the same thread. */
const char *fa_last_error(void);

/* ABI version of this library (major * 100 + minor). */
int fa_version(void);

/* Failure detection.  Every wait inside the tensor-core kernels (bf16, e4m3,
 * fp32 on the tensor cores) is bounded (two seconds); a wait that runs out
 * makes the kernel abandon its work, drain its copies and MMAs, free its
 * tensor memory and return, and sets a device status word, so that the
 * context stays usable.  fa_device_status synchronises `stream` (a
 * cudaStream_t, NULL = legacy default stream), reads and clears those words,
 * and returns FA_ETIMEOUT if a wait ran out since the previous check (the
 * outputs of the calls in between are then not valid), FA_OK otherwise, or
 * FA_ECUDA if the reads fail. */
fa_status fa_device_status(void *stream);

/* Test hook for the path above, off by default: while enabled, CTA 0 of each
 * tensor-core kernel launch skips one of its loads, so that a bounded wait
 * runs out.  Not for production use. */
fa_status fa_test_drop_arrive(int enable);

/* Test hook, off by default (n = 0): while n > 0, the persistent launches of
 * the tensor-core kernels (bf16 / e4m3 prefill and variable-length batches)
 * use at most n CTAs, so that each CTA walks more units.  Results must not
 * depend on it: a row's arithmetic is the same whichever CTA or slot runs it
 * ("FlashAttention forward in C", section 4: the thread-pool result equals
 * the serial one bit for bit).  FA_EINVAL for n < 0.  Host-side state of the
 * process, not thread-safe.  Not for production use. */
fa_status fa_test_max_ctas(int64_t n);

#ifdef __cplusplus
}
#endif

#endif /* FA_GB300_FA_H */
