/*
 * fa.h — C ABI of the exact-attention library for one NVIDIA GB300 (sm_103a).
 *
 * The library computes exact scaled-dot-product attention
 *
 *     O = softmax(scale * Q K^T) V
 *
 * FlashAttention-2 style: an outer loop over 128-row query blocks and an inner
 * loop over key/value blocks (64 rows for D <= 64, 128 for D = 128 in the
 * forward pass) with an online softmax (running row
 * maximum m and running sum l), so the [S, S] score matrix never reaches
 * memory.  Only O and the per-row logsumexp L are written.  The backward pass
 * recomputes the probabilities from L.  Definitions followed:
 *   - forward recurrence and L: "从零训练语言模型（第二部分：FlashAttention 与设备内存）"
 *     §安全 / 在线 softmax and §使用 LSE 连接正向和反向传播;
 *     "T5 讲解：FlashAttention forward" §④ (online softmax update), §⑤ (causal
 *     block skipping), §⑥ (default scale 1/sqrt(D));
 *   - backward: the same "第二部分" page §反向传播 (P = exp(S - L), dV = P^T dO,
 *     dP = dO V^T, dS = P o (dP - D), dQ = dS K * scale, dK = dS^T Q * scale),
 *     and the CS336 Assignment 2 write-up, "4. Problem (flash_backward)"
 *     (recompute backward with the row vector D = rowsum(dO o O)).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * Layout: every matrix argument (q, k, v, o, dout, dq, dk, dv) is a dense,
 *   contiguous row-major tensor [B, H, S, D] of 16-bit floats (fp16 or bf16,
 *   chosen by `dtype`), element strides (H*S*D, S*D, D, 1).  Query and key
 *   lengths are equal (S).  `lse` is fp32 [B, H, S]; it holds the NATURAL-log
 *   logsumexp of the scaled scores, L_i = ln sum_j exp(scale * q_i . k_j).
 * Causal: when `causal` is nonzero, query i attends to keys j <= i (top-left
 *   aligned mask).  Every query row then sees at least key 0.
 * Scale: any finite float; the usual value is 1/sqrt(D).
 * Supported: D in {16, 32, 64, 128}; S >= 0; B, H >= 0; B*H < 2^31;
 *   S < 2^31.  S == 0 or B*H == 0 is a valid empty call that launches nothing.
 * Pointers: DEVICE pointers of the current CUDA device, each 16-byte aligned
 *   (the tensor-memory-access engine requires it).  In an empty call they are
 *   not used and may be NULL.
 * Ownership: the caller owns every buffer and the stream.  The library
 *   allocates no memory, keeps no pointer after a call returns, and does not
 *   synchronise: results are ready when `stream` reaches the launched work.
 * Stream: a cudaStream_t passed as void* (NULL = the legacy default stream).
 * Errors: every entry point validates all arguments before launching anything
 *   and returns FA_OK or an fa_status code; nothing is launched on error.
 *   fa_last_error_detail() gives a one-line description of the last failure
 *   on the calling thread.  Kernels never trap: a device-side pipeline wait
 *   that exceeds its time limit (2 s by default, see fa_set_wait_limit_ns)
 *   ends the kernel and sets a device error word that fa_check_device_errors()
 *   reads.
 */
#ifndef FA_GB300_H
#define FA_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  FA_OK = 0,
  FA_ERR_INVALID_ARG = 1, /* null pointer, negative size, non-finite scale, bad dtype */
  FA_ERR_UNSUPPORTED = 2, /* head dimension not in {16,32,64,128}, or sizes too large */
  FA_ERR_ALIGNMENT = 3,   /* a pointer is not 16-byte aligned */
  FA_ERR_WORKSPACE = 4,   /* workspace missing or smaller than fa_bwd_workspace_size() */
  FA_ERR_CUDA = 5,        /* a CUDA runtime/driver call or a kernel launch failed */
  FA_ERR_TIMEOUT = 6      /* a device pipeline wait exceeded its limit (see fa_check_device_errors) */
} fa_status;

typedef enum { FA_FP16 = 0, FA_BF16 = 1 } fa_dtype;

/*
 * Forward pass.
 *   q, k, v : [B, H, S, D] inputs (read only).
 *   o       : [B, H, S, D] output, same dtype; O = softmax(scale Q K^T (+mask)) V.
 *   lse     : [B, H, S] fp32 output, natural-log logsumexp per query row.
 * Per query block the kernel visits only key blocks that are not wholly above
 * the diagonal when causal ("T5 讲解" §⑤), masks element-wise only in the
 * diagonal block and in a ragged last key block, and writes O / l and
 * L = m + ln l in the epilogue.
 */
fa_status fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int64_t B, int64_t H,
                 int64_t S, int64_t D, int causal, float scale, fa_dtype dtype, void* stream);

/*
 * Forward pass with grouped K/V heads (multi-query / grouped-query attention,
 * "Inside FlashAttention" §6.1, the MQA / GQA interface: several query heads
 * share one K/V head, and K, V are passed with fewer heads instead of being
 * copied out to H heads).
 *   q, o    : [B, H, S, D];  lse : [B, H, S] fp32.
 *   k, v    : [B, H_kv, S, D].
 * H must be a positive multiple of H_kv (H_kv >= 1); query head h of batch b
 * reads K/V head h / (H / H_kv) of batch b, so each K/V head serves a run of
 * H / H_kv consecutive query heads.  H_kv = H is fa_fwd; H_kv = 1 is
 * multi-query attention.  A call with B*H == 0 (then H_kv == 0 is allowed
 * when H == 0) or S == 0 launches nothing.  Every other convention
 * (layout, alignment, ownership, errors) is fa_fwd's; a bad H_kv returns
 * FA_ERR_INVALID_ARG.
 */
fa_status fa_fwd_gqa(const void* q, const void* k, const void* v, void* o, float* lse, int64_t B, int64_t H,
                     int64_t H_kv, int64_t S, int64_t D, int causal, float scale, fa_dtype dtype, void* stream);

/*
 * Bytes of device workspace fa_bwd needs for these sizes: the fp32 row vector
 * D_i = rowsum(dO o O) for every (b, h, i), rounded up to 256 bytes.
 */
size_t fa_bwd_workspace_size(int64_t B, int64_t H, int64_t S, int64_t D);

/*
 * Backward pass (recompute).  Given the forward inputs, its outputs o and lse,
 * and the loss gradient dout = dL/dO, writes dq, dk, dv ([B, H, S, D], same
 * dtype).  Three passes run in order on `stream`:
 *   1. D_i = rowsum(dO o O) into the workspace (fp32);
 *   2. per 128-key block: dV = sum_i P^T dO and dK = scale * sum_i dS^T Q over the
 *      query blocks that see it, P = exp(S - L) recomputed from lse;
 *   3. per 128-query block: dQ = scale * sum_j dS K over its visible key blocks.
 * At D <= 64 the dQ kernel computes D_i itself (and writes it to the
 * workspace): two kernels then run, the dQ pass first and the dK/dV pass after.
 * workspace: device buffer of at least fa_bwd_workspace_size() bytes, 256-byte
 * aligned, owned by the caller; its contents on entry do not matter.
 */
fa_status fa_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout,
                 const float* lse, void* dq, void* dk, void* dv, int64_t B, int64_t H, int64_t S, int64_t D,
                 int causal, float scale, fa_dtype dtype, void* workspace, size_t workspace_bytes,
                 void* stream);

/*
 * fa_bwd with timing marks.  Same arguments, same launches, same results;
 * in addition, each non-NULL entry of `marks` (a cudaEvent_t passed as void*,
 * owned by the caller) is recorded on `stream`, in this order: marks[0]
 * before the first kernel; marks[1] after the Delta kernel, or after the dQ
 * kernel where that computes Delta (fa_bwd, fa_bwd_gqa at D <= 64; the
 * window and packed-batch calls always run the Delta kernel); marks[2] after
 * the dK/dV kernel (and its partial-sum reduction); marks[3] after the dQ
 * kernel where it runs last, else right after marks[2].  Lets a caller time
 * each kernel with CUDA events on the stream that runs it.  `marks` itself
 * may be NULL.
 */
fa_status fa_bwd_marked(const void* q, const void* k, const void* v, const void* o, const void* dout,
                        const float* lse, void* dq, void* dk, void* dv, int64_t B, int64_t H, int64_t S,
                        int64_t D, int causal, float scale, fa_dtype dtype, void* workspace,
                        size_t workspace_bytes, void* stream, void* const* marks);

/*
 * Backward pass with grouped K/V heads: the gradient of fa_fwd_gqa.
 *   q, o, dout, dq : [B, H, S, D];  lse : [B, H, S] fp32.
 *   k, v, dk, dv   : [B, H_kv, S, D].
 * A K/V head's gradients sum the contributions of all H / H_kv query heads
 * that read it: dV_g = sum over the group's heads h of P_h^T dO_h, and dK_g
 * likewise with dS_h^T Q_h.  A dK/dV CTA owns one (K/V head, 128-key block)
 * and streams query heads of the group one after another through the same
 * accumulators.  When the K/V heads alone give too few CTAs to fill the GPU
 * (few K/V heads, short sequences), s CTAs share a (K/V head, key block),
 * each over G/s of the group's heads (s the smallest divisor of G that gives
 * 304 CTAs, else G); they write fp32 partial sums to the workspace and a
 * further kernel adds them in a fixed order.  No atomics either way: results
 * are deterministic.  Workspace: fa_bwd_gqa_workspace_size() bytes.  Other
 * conventions as fa_bwd; H_kv as in fa_fwd_gqa.
 */
fa_status fa_bwd_gqa(const void* q, const void* k, const void* v, const void* o, const void* dout,
                     const float* lse, void* dq, void* dk, void* dv, int64_t B, int64_t H, int64_t H_kv,
                     int64_t S, int64_t D, int causal, float scale, fa_dtype dtype, void* workspace,
                     size_t workspace_bytes, void* stream);

/*
 * Bytes of device workspace fa_bwd_gqa needs: the fp32 row vector D of every
 * query row (B*H*S floats, rounded up to 256 bytes), plus, when the dK/dV
 * pass splits the group (see fa_bwd_gqa), s * B*H_kv*S*2*D fp32 partial sums
 * (rounded up to 256 bytes).  Equals fa_bwd_workspace_size() when H_kv = H.
 * Returns 0 for an empty problem or an H_kv that does not divide H.
 */
size_t fa_bwd_gqa_workspace_size(int64_t B, int64_t H, int64_t H_kv, int64_t S, int64_t D);

/* fa_bwd_gqa with the timing marks of fa_bwd_marked (marks[2] is recorded
 * after the dK/dV kernel and, when it runs, the partial-sum kernel). */
fa_status fa_bwd_gqa_marked(const void* q, const void* k, const void* v, const void* o, const void* dout,
                            const float* lse, void* dq, void* dk, void* dv, int64_t B, int64_t H, int64_t H_kv,
                            int64_t S, int64_t D, int causal, float scale, fa_dtype dtype, void* workspace,
                            size_t workspace_bytes, void* stream, void* const* marks);

/*
 * Sliding-window (local) attention ("Inside FlashAttention" §6.1, window_size
 * = (left, right): only the key blocks inside the window are computed).  Key j
 * is visible to query i only if i - window_left <= j <= i + window_right; a
 * negative side is unlimited, and `causal` additionally hides j > i (so
 * causal with (left, 0) is the usual local causal window).  Layouts, grouped
 * heads (H_kv) and every other convention as fa_fwd_gqa / fa_bwd_gqa.  Each
 * 128-row query tile (or 128-key tile in the backward) visits only the key
 * (query) blocks that meet its band; blocks crossing either edge of the band
 * are masked element-wise, the others run unmasked.  Every query row sees at
 * least its own key, so no row is empty.  A window that covers the whole
 * sequence runs the ordinary kernels.  Workspace: fa_bwd_gqa_workspace_size().
 */
fa_status fa_fwd_window(const void* q, const void* k, const void* v, void* o, float* lse, int64_t B, int64_t H,
                        int64_t H_kv, int64_t S, int64_t D, int causal, int64_t window_left, int64_t window_right,
                        float scale, fa_dtype dtype, void* stream);

fa_status fa_bwd_window(const void* q, const void* k, const void* v, const void* o, const void* dout,
                        const float* lse, void* dq, void* dk, void* dv, int64_t B, int64_t H, int64_t H_kv,
                        int64_t S, int64_t D, int causal, int64_t window_left, int64_t window_right, float scale,
                        fa_dtype dtype, void* workspace, size_t workspace_bytes, void* stream);

/* fa_bwd_window with the timing marks of fa_bwd_marked. */
fa_status fa_bwd_window_marked(const void* q, const void* k, const void* v, const void* o, const void* dout,
                               const float* lse, void* dq, void* dk, void* dv, int64_t B, int64_t H, int64_t H_kv,
                               int64_t S, int64_t D, int causal, int64_t window_left, int64_t window_right,
                               float scale, fa_dtype dtype, void* workspace, size_t workspace_bytes, void* stream,
                               void* const* marks);

/*
 * Split-KV forward with a logsumexp merge ("T5 讲解" §⑥: the stored
 * L = m + log l is what lets shards be merged).  The keys are cut into shards
 * of ceil(S / num_splits) keys rounded up to a multiple of 128; one launch
 * computes, per (b, h, query tile, shard), the fp32 output normalised over the
 * shard's keys and its logsumexp into `workspace`, and a second kernel merges
 * the shards:  L = ln sum_s exp(L_s),  O = sum_s exp(L_s - L) O_s.  The result
 * equals fa_fwd_gqa's up to fp32 rounding; it pays off where B*H*ceil(S/512)
 * (ceil(S/256) for D = 128) query tiles alone cannot fill the GPU.  Layouts,
 * heads and causal as in fa_fwd_gqa.  num_splits >= 1 (1 is legal: one
 * shard); fa_splitkv_num_splits() proposes one.  workspace: at least
 * fa_fwd_splitkv_workspace_size() bytes, 256-byte aligned, owned by the caller.
 */
fa_status fa_fwd_splitkv(const void* q, const void* k, const void* v, void* o, float* lse, int64_t B, int64_t H,
                         int64_t H_kv, int64_t S, int64_t D, int causal, int64_t num_splits, float scale,
                         fa_dtype dtype, void* workspace, size_t workspace_bytes, void* stream);

/* Workspace of fa_fwd_splitkv: shards * B*H*S * (D + 1) fp32 values, rounded up to 256 bytes. */
size_t fa_fwd_splitkv_workspace_size(int64_t B, int64_t H, int64_t S, int64_t D, int64_t num_splits);

/* A split count that gives a 152-SM GPU at least two CTAs per SM (1 when the
 * query tiles already do; at most one shard per 128 keys). */
int64_t fa_splitkv_num_splits(int64_t B, int64_t H, int64_t S, int64_t D);

/*
 * The merge on its own, for partials computed elsewhere (other GPUs' key
 * shards, a cache of earlier keys):
 *   o_part   : DEVICE fp32 [shards, rows, D], each shard's normalised output;
 *   lse_part : DEVICE fp32 [shards, rows], each shard's natural-log L_s
 *              (-inf for a row that sees no key of the shard; its O_s is ignored);
 *   o        : [rows, D] 16-bit output (dtype);  lse : [rows] fp32 output.
 * A row whose every L_s is -inf gets O = 0 and L = -inf.  D in {16,32,64,128}.
 */
fa_status fa_merge_lse(const float* o_part, const float* lse_part, void* o, float* lse, int64_t shards,
                       int64_t rows, int64_t D, fa_dtype dtype, void* stream);

/*
 * Packed variable-length batches ("Inside FlashAttention" §6.1, varlen: samples
 * of different lengths concatenated with no padding, a prefix-sum array
 * cu_seqlens marking their bounds, and no attention across samples).
 *   q, o           : [T, H, D]     (token-major; T = total tokens)
 *   k, v           : [T, H_kv, D]  (H a positive multiple of H_kv, as in fa_fwd_gqa)
 *   lse            : [H, T] fp32, natural-log logsumexp
 *   cu_seqlens     : DEVICE int32 [batch + 1]; cu[0] = 0, non-decreasing,
 *                    cu[batch] <= total; sample b is tokens cu[b] .. cu[b+1]-1
 *                    (empty samples allowed) and attends only to itself, with the
 *                    top-left causal mask inside the sample when causal.
 *   max_seqlen     : host bound on every sample length (sizes the grid).
 * The kernels read cu_seqlens themselves.  A sample longer than max_seqlen,
 * or one that runs past `total`, is not computed: the kernels record it and
 * fa_check_device_errors() then returns FA_ERR_INVALID_ARG.  Rows of tokens
 * that no sample covers are left unwritten.  Other conventions as fa_fwd
 * (cu_seqlens needs 4-byte alignment only).  batch, H, max_seqlen or total
 * equal to 0 is an empty call.
 */
fa_status fa_fwd_varlen(const void* q, const void* k, const void* v, void* o, float* lse,
                        const int32_t* cu_seqlens, int64_t batch, int64_t max_seqlen, int64_t total, int64_t H,
                        int64_t H_kv, int64_t D, int causal, float scale, fa_dtype dtype, void* stream);

/* Workspace bytes of fa_bwd_varlen: Delta for the T*H query rows, plus the
 * dK/dV partial sums when the grouped pass splits (as fa_bwd_gqa_workspace_size,
 * with batch entries of up to max_seqlen rows; T*H_kv K/V rows). */
size_t fa_bwd_varlen_workspace_size(int64_t batch, int64_t max_seqlen, int64_t total, int64_t H, int64_t H_kv,
                                    int64_t D);

/* Backward of fa_fwd_varlen: dq [T, H, D], dk, dv [T, H_kv, D]; the packed
 * layout and checks of fa_fwd_varlen, the rest as fa_bwd_gqa. */
fa_status fa_bwd_varlen(const void* q, const void* k, const void* v, const void* o, const void* dout,
                        const float* lse, void* dq, void* dk, void* dv, const int32_t* cu_seqlens, int64_t batch,
                        int64_t max_seqlen, int64_t total, int64_t H, int64_t H_kv, int64_t D, int causal,
                        float scale, fa_dtype dtype, void* workspace, size_t workspace_bytes, void* stream);

/* fa_bwd_varlen with the timing marks of fa_bwd_marked. */
fa_status fa_bwd_varlen_marked(const void* q, const void* k, const void* v, const void* o, const void* dout,
                               const float* lse, void* dq, void* dk, void* dv, const int32_t* cu_seqlens,
                               int64_t batch, int64_t max_seqlen, int64_t total, int64_t H, int64_t H_kv, int64_t D,
                               int causal, float scale, fa_dtype dtype, void* workspace, size_t workspace_bytes,
                               void* stream, void* const* marks);

/*
 * fa_bwd without a workspace argument, for callers that cannot allocate
 * device memory when they run the backward pass (for example code inside a
 * custom allocator or a fully carved-up memory pool, or a framework that
 * forbids cudaMalloc on its hot path).  The pages describe no such variant:
 * it has no counterpart there.
 *
 * Same arguments and results as fa_bwd minus the workspace.  The scratch row
 * vector D lives in a fixed device array inside the library (8 MiB, held by
 * every GPU that loads the library until the process exits), so
 * B*H*S may not exceed 2^21 rows; larger calls return FA_ERR_UNSUPPORTED.
 * The call allocates nothing: no cudaMalloc, cudaFree or allocating library
 * routine.  Its first call on a device looks up the array's device address
 * (with that device current) and caches it; make that first call before any
 * stream capture.  All calls share the one array and it keeps the last
 * call's contents (each call overwrites the rows it uses before reading
 * them): calls whose work overlaps on the GPU, e.g. on two streams at once,
 * race on it and must be serialised by the caller.
 */
fa_status fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const void* dout,
                         const float* lse, void* dq, void* dk, void* dv, int64_t B, int64_t H, int64_t S,
                         int64_t D, int causal, float scale, fa_dtype dtype, void* stream);

/* Static, human-readable name of a status code. */
const char* fa_status_string(fa_status status);

/* One-line description of the last failure on the calling thread ("" if none). */
const char* fa_last_error_detail(void);

/*
 * Synchronises `stream`, then reads and clears the device error word that the
 * kernels set when a pipeline wait times out or a packed batch's cu_seqlens
 * contradicts its call.  Returns FA_ERR_TIMEOUT or FA_ERR_INVALID_ARG (the
 * latter for cu_seqlens) if it was set, FA_ERR_CUDA if the synchronisation
 * failed, else FA_OK.  Meant for
 * tests and debugging; the compute entry points never synchronise.
 */
fa_status fa_check_device_errors(void* stream);

/*
 * Sets the time limit, in nanoseconds, of every pipeline wait in the kernels
 * launched after this call (a wait on a barrier that another warp of the same
 * CTA completes: operands landed, scores computed, a stage freed).  0 restores
 * the default of 2 s.  Returns the previous limit.  Process-wide, not tied to
 * a stream or device.  A wait that runs past its limit makes its CTA stop
 * early: it drains its own copies and MMAs (those waits keep the 2 s limit),
 * frees its tensor memory and exits, and fa_check_device_errors() returns
 * FA_ERR_TIMEOUT; the outputs of that call are then undefined.  A limit far
 * below the kernels' own latencies (nanoseconds) makes that happen on purpose,
 * which is how the tests exercise this path.  Not part of the pages' interface:
 * failure handling for callers that must not hang.
 */
uint64_t fa_set_wait_limit_ns(uint64_t ns);

#ifdef __cplusplus
}
#endif

#endif /* FA_GB300_H */
