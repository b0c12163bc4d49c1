/*
 * fa.h — C ABI of the GB300 (sm_103a) fused attention library (libfa.so).
 *
 * Exact scaled-dot-product attention
 *     O = softmax(scale * Q K^T [+ causal mask]) V
 * computed as one fused, tiled forward kernel with an online softmax that
 * saves the per-row log-sum-exp, and a recompute-based backward that rebuilds
 * P from Q, K and that log-sum-exp. No N x N matrix is ever written to memory.
 *
 * Sources (web pages, cited by title and section):
 *  - "transformer模型详解（十）：FlashAttention优化技术" (Transformer explained,
 *    part 10: FlashAttention), sections "Kernel Fusion：消灭中间落盘" (one kernel,
 *    only the final output written), "Tiling 分块策略：匹配硬件极限" (B_q x B_k
 *    tiles in on-chip memory; online softmax: per-tile max and exp-sum, update
 *    of the global max with rescaling, one final normalisation),
 *    "Re-computation 而非缓存" (backward: outer loop over K/V column blocks,
 *    inner loop over Q row blocks, scores and probabilities recomputed) and
 *    "硬件依赖不可忽视" (sequence length a multiple of 16, head dimension
 *    preferably 64/128/256). Its AMP example calls flash_attn_func(q, k, v).
 *  - "在TPU上移植Flash Attention的工程实践与挑战", Example 2 (chunked attention):
 *    tensors laid out (batch, heads, seq, head_dim).
 *
 * Conventions shared by every entry point
 *  - Tensors q, k, v, o, dO, dq, dk, dv: dense, contiguous [B, H, N, d] in the
 *    element type given by `dtype` (fp16 or bf16), row pitch d elements.
 *    lse: fp32 [B, H, N], natural-log log-sum-exp of the scaled logits.
 *  - All data pointers are DEVICE pointers owned by the caller; the library
 *    allocates nothing on these paths. Every pointer must be 16-byte aligned
 *    (a TMA requirement), else FA_ERR_ALIGNMENT.
 *  - Supported shapes: d in {64, 128, 256}; any N >= 1 (a last tile that
 *    runs past N is zero-filled on load, masked, and not stored); B, H >= 1;
 *    B*H*N' < 2^31 with N' = N rounded up to 128; N <= 65535*128 =
 *    8,388,480 (one backward CTA column per 128-key block, and a grid's y
 *    extent is at most 65535). Anything else: FA_ERR_UNSUPPORTED, no launch.
 *  - scale: finite and > 0, else FA_ERR_INVALID_ARG. The pages use
 *    scale = d^-1/2.
 *  - causal != 0: query i attends to keys j <= i.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *    stream). Work is enqueued asynchronously; argument errors are returned
 *    synchronously with nothing enqueued; a failed launch returns FA_ERR_CUDA.
 *  - Device-side problems (a bounded wait that timed out, a failed index
 *    check) do not trap: they are recorded in a device status word that
 *    fa_device_status() reads and clears.
 *  - The current CUDA device must be a compute capability 10.3 GPU (sm_103a
 *    code only), else FA_ERR_UNSUPPORTED.
 */
#ifndef FA_H_
#define FA_H_

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  FA_OK = 0,
  FA_ERR_INVALID_ARG = 1,  /* null pointer, bad scale, bad enum value */
  FA_ERR_UNSUPPORTED = 2,  /* shape/dtype/device outside the supported set */
  FA_ERR_ALIGNMENT = 3,    /* a pointer is not 16-byte aligned */
  FA_ERR_WORKSPACE = 4,    /* workspace missing or smaller than fa_bwd_workspace_size() */
  FA_ERR_CUDA = 5,         /* a CUDA runtime/driver call failed */
  FA_ERR_TIMEOUT = 6,      /* a device-side bounded wait expired (from fa_device_status) */
  FA_ERR_DEVICE_FAULT = 7  /* a device-side check failed (from fa_device_status) */
} fa_status;

typedef enum { FA_F16 = 0, FA_BF16 = 1 } fa_dtype;

/*
 * Forward pass (page 2, "Kernel Fusion" + "Tiling" + online softmax).
 *   in : q, k, v  [B,H,N,d] dtype
 *   out: o        [B,H,N,d] dtype  = softmax(scale*q k^T [causal]) v, rounded to dtype
 *        lse      [B,H,N]   fp32   = ln(sum_j exp(scale * q_i . k_j)) over visible j
 * One kernel launch. o and lse are written in full.
 */
fa_status fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int d,
                 float scale, int causal, fa_dtype dtype, void* stream);

/*
 * fa_fwd that also writes o_lo [B,H,N,d] dtype = dtype(O_fp32 - float(o)), the
 * rounding residual of the stored output (same kernel, same o and lse). Passed
 * to fa_bwd, o + o_lo restores O to fp32 accuracy for D = rowsum(dO * O).
 * That matters when rows are nearly one-hot: dP - D then cancels, and the
 * output rounding of o alone would leak into dS (the pages fix no precision for
 * this step; see the backward's contract). o_lo NULL behaves as fa_fwd.
 * o_lo must be 16-byte aligned.
 */
fa_status fa_fwd_ex(const void* q, const void* k, const void* v, void* o, float* lse, void* o_lo, int B, int H, int N,
                    int d, float scale, int causal, fa_dtype dtype, void* stream);

/*
 * Options beyond plain multi-head attention, for fa_fwd_opt / fa_bwd_opt.
 * Zero-initialise, then set what is needed; a NULL options pointer means all
 * defaults (then the _opt calls equal fa_fwd_ex / fa_bwd).
 *  - n_kv_heads: K and V (and dK, dV) have this many heads, [B, n_kv_heads,
 *    N, d]; query head h reads K/V head h / (H / n_kv_heads) (grouped-query
 *    attention; 1 is multi-query attention, as in the multi-query kernel of
 *    page "高级特性：探索PyTorch/XLA的Pallas内核和Flash Attention实现", section
 *    "Pallas内核：自定义高效计算的关键"). 0 means H. H must be a multiple of
 *    it (else FA_ERR_UNSUPPORTED); negative: FA_ERR_INVALID_ARG. In the
 *    backward dK, dV of a K/V head are summed over its H / n_kv_heads query
 *    heads inside one CTA (no atomics; dk, dv stay bitwise reproducible).
 *  - kv_len: NULL, or a DEVICE int32 array [B] (4-byte aligned, else
 *    FA_ERR_ALIGNMENT): in batch b every query sees only keys j < kv_len[b]
 *    (a key-padding mask; the masking use of an attention bias on page
 *    "transformer模型详解（十）：FlashAttention优化技术", section "精度与稳定性的平衡").
 *    Values are clamped to [0, N] on the device. Combined with causal, query
 *    i sees keys j <= i with j < kv_len[b]. A query that sees no key
 *    (kv_len[b] = 0) gets O = 0 and LSE = -inf, and contributes zero
 *    gradients. Key tiles wholly past kv_len[b] are skipped by the forward.
 *  - o_fp32: nonzero: O is fp32 [B,H,N,d] (the forward writes it so, unrounded;
 *    the backward reads it so), the mixed-precision output of page
 *    "在TPU上移植Flash Attention的工程实践与挑战", Example 3 (16-bit inputs and
 *    products, fp32 result). o_lo must then be NULL (FA_ERR_INVALID_ARG).
 *  - dq_mode (backward only): how dQ = scale * dS K is formed (page
 *    "transformer模型详解（十）：FlashAttention优化技术", section "Re-computation
 *    而非缓存", accumulates dq across the K/V block loop).
 *      FA_DQ_ACCUMULATE: the key-major main kernel adds fp32 partial tiles into
 *        the workspace's dQ accumulator (bulk reductions), and a conversion pass
 *        scales and rounds it; dq's summation order depends on scheduling.
 *      FA_DQ_SEPARATE: the main kernel computes dK, dV only; a query-major pass
 *        recomputes S and dP per 128 x 128 tile and keeps dQ in tensor memory
 *        (no accumulator, no zeroing, dq bitwise reproducible); d = 64 and 128
 *        only (else FA_ERR_UNSUPPORTED).
 *      FA_DQ_DEFAULT (0): the library picks the faster of the two for the
 *        head dimension and mask, as measured on GB300 (the table is in the
 *        design notes).
 *    Other values: FA_ERR_INVALID_ARG.
 */
enum { FA_DQ_DEFAULT = 0, FA_DQ_ACCUMULATE = 1, FA_DQ_SEPARATE = 2 };
typedef struct fa_options {
  int n_kv_heads;
  const int* kv_len;
  int o_fp32;
  int dq_mode;
} fa_options;

/* Forward with options: arguments and results as fa_fwd_ex, k and v with
 * opt->n_kv_heads heads, o in fp32 when opt->o_fp32. */
fa_status fa_fwd_opt(const void* q, const void* k, const void* v, void* o, float* lse, void* o_lo, int B, int H,
                     int N, int d, float scale, int causal, fa_dtype dtype, const fa_options* opt, void* stream);

/*
 * Forward with the key range of each query block split over several CTAs
 * (page "transformer模型详解（十）：FlashAttention优化技术", section "Tiling
 * 分块策略": the running max and sum of the online softmax are updated block by
 * block, so disjoint key ranges can be reduced apart and joined afterwards).
 * Each of the kv_splits ranges writes a normalised fp32 partial O_s and LSE_s
 * to the workspace; a second launch joins them, LSE = ln sum_s e^(LSE_s),
 * O = sum_s e^(LSE_s - LSE) O_s, and writes o (with o_lo when given, or fp32
 * with opt->o_fp32) and lse, with the same meaning as fa_fwd_opt. It pays where
 * the grid would otherwise leave SMs idle (few heads, short sequences).
 *  - kv_splits: 1 = no split (exactly fa_fwd_opt; workspace unused); 2..16 =
 *    that many ranges; 0 = the library's choice, fa_fwd_kv_splits(); above 16:
 *    FA_ERR_UNSUPPORTED.
 *  - workspace: device memory of fa_fwd_workspace_size(B,H,N,d,kv_splits)
 *    bytes, 256-byte aligned, caller-owned (contents on entry do not matter);
 *    may be NULL when kv_splits resolves to 1.
 * fa_fwd_workspace_size returns 0 for kv_splits < 2 (no workspace) and for
 * unsupported shapes.
 */
fa_status fa_fwd_split(const void* q, const void* k, const void* v, void* o, float* lse, void* o_lo, int B, int H,
                       int N, int d, float scale, int causal, fa_dtype dtype, const fa_options* opt, int kv_splits,
                       void* workspace, size_t workspace_bytes, void* stream);
int fa_fwd_kv_splits(int B, int H, int N, int d, int causal);
size_t fa_fwd_workspace_size(int B, int H, int N, int d, int kv_splits);

/*
 * Query tiles of 128 rows that one CTA of the forward (without a split) takes
 * as one work item for this shape: 2 (the two softmax warpgroups take turns on
 * the tensor core) or 1 (twice the items, each half as long: short rows and few
 * heads, where two-tile items would leave SMs idle or make the longest item the
 * critical path). The library picks it on every forward call; the result does
 * not depend on it (each query row's computation is the same). d = 256 always
 * takes 1. Returns 0 for an unsupported shape.
 */
int fa_fwd_tiles_per_item(int B, int H, int N, int d, int causal);

/*
 * Bytes of device workspace fa_bwd needs: fp32 D [B,H,Np], fp32 LSE*log2(e)
 * [B,H,Np] and the fp32 dQ accumulator [B,H,Np,d], each 256-byte aligned,
 * with Np = N rounded up to 128 (each head's rows padded so that every query
 * step or tile of the backward starts aligned and stays in its head). The
 * separate dQ pass leaves the accumulator untouched.
 * Returns 0 for unsupported shapes.
 */
size_t fa_bwd_workspace_size(int B, int H, int N, int d);

/*
 * Backward pass (page 2, "Re-computation"): from the forward's o and lse and
 * the upstream gradient dO, computes
 *   D  = rowsum(dO * O), O = o + o_lo        (fp32, workspace; O = o if o_lo is NULL)
 *   P  = exp(scale * q k^T - lse)            (recomputed per tile, never stored)
 *   dV = P^T dO;  dP = dO v^T;  dS = P * (dP - D)
 *   dQ = scale * dS k;  dK = scale * dS^T q
 * d is 64, 128 or 256 (for d = 256 each 128-key block makes two passes, one
 * per half of the head dimension, recomputing S and dP in each).
 * o_lo: NULL, or the residual written by fa_fwd_ex for this o.
 * Writes dq, dk, dv [B,H,N,d] dtype in full (no accumulate-into). Three
 * launches on `stream`: preprocess (D, LSE*log2e, zero the fp32 dQ
 * accumulator), the main kernel (one CTA per 128-key tile, dQ partial tiles
 * added into the accumulator with bulk reductions), and the dQ conversion.
 * Summation order of dQ depends on scheduling, so dq is not bitwise
 * reproducible; dk, dv are.
 * workspace: device memory of at least fa_bwd_workspace_size(B,H,N,d) bytes,
 * caller-owned, 256-byte aligned; its contents on entry do not matter.
 */
fa_status fa_bwd(const void* q, const void* k, const void* v, const void* o, const void* dO, const float* lse,
                 void* dq, void* dk, void* dv, const void* o_lo, void* workspace, size_t workspace_bytes, int B, int H,
                 int N, int d, float scale, int causal, fa_dtype dtype, void* stream);

/* Backward with options: arguments and results as fa_bwd; k, v, dk, dv with
 * opt->n_kv_heads heads; o in fp32 when opt->o_fp32; the same kv_len as the
 * forward that produced o and lse. The workspace is sized by H (query heads). */
fa_status fa_bwd_opt(const void* q, const void* k, const void* v, const void* o, const void* dO, const float* lse,
                     void* dq, void* dk, void* dv, const void* o_lo, void* workspace, size_t workspace_bytes, int B,
                     int H, int N, int d, float scale, int causal, fa_dtype dtype, const fa_options* opt,
                     void* stream);

/*
 * fa_bwd for callers that cannot allocate device memory: the workspace is a
 * fixed array inside this library instead of caller memory. The pages have no
 * counterpart; this entry point exists only for how the library is called.
 * It is meant for code that runs where allocating is not allowed or not wise:
 * an inference runtime's plugin hook or a framework extension point whose
 * contract forbids allocation while enqueuing work, or a process whose device
 * memory is owned by another allocator (cudaMalloc may also synchronise).
 * Same arguments and results as fa_bwd, minus the workspace. Limits and rules:
 *  - problems whose fa_bwd_workspace_size() exceeds FA_NOALLOC_SCRATCH_BYTES
 *    (64 MiB; for d = 128 that is B*H*N up to about 129,000 rows) return
 *    FA_ERR_WORKSPACE with nothing enqueued;
 *  - the array is device memory of the library's own module, one 64 MiB copy
 *    per CUDA context. Under lazy module loading (the CUDA default) a context
 *    gets its copy at the first fa_bwd_noalloc call made in it: that first
 *    call loads the module and so allocates the 64 MiB (through the driver).
 *    Make it at set-up time, outside the path that must not allocate and
 *    before any stream capture. Under CUDA_MODULE_LOADING=EAGER every context
 *    that loads the library gets its copy when the context is created, whether
 *    or not it ever calls this entry point. The copy lasts as long as the
 *    context;
 *  - every call looks up the current device's copy (a host-side lookup once
 *    the module is loaded), so a context re-created after cudaDeviceReset is
 *    served from its own new copy;
 *  - all calls share the array: calls whose GPU work can overlap (different
 *    streams without ordering) race on it and must be serialised by the caller.
 * Calls no cudaMalloc/cudaFree and no allocating library routine.
 */
#define FA_NOALLOC_SCRATCH_BYTES (64ull << 20)
fa_status fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const void* dO,
                         const float* lse, void* dq, void* dk, void* dv, const void* o_lo, int B, int H, int N, int d,
                         float scale, int causal, fa_dtype dtype, void* stream);

/*
 * The phases of fa_bwd as separate calls (same arguments and rules), exposed
 * so each kernel can be timed on its own. fa_bwd is fa_bwd_preprocess followed
 * by fa_bwd_main with dq given. fa_bwd_main's dq is optional: given, the dQ
 * conversion is enqueued right after the main kernel, so dq is complete when
 * the call's work completes; NULL, dQ is left (unscaled, fp32) in the
 * workspace and fa_bwd_dq_convert turns it into dq afterwards.
 */
fa_status fa_bwd_preprocess(const void* o, const void* o_lo, const void* dO, const float* lse, void* workspace,
                            size_t workspace_bytes, int B, int H, int N, int d, fa_dtype dtype, void* stream);
fa_status fa_bwd_main(const void* q, const void* k, const void* v, const void* dO, void* dk, void* dv, void* dq,
                      void* workspace, size_t workspace_bytes, int B, int H, int N, int d, float scale, int causal,
                      fa_dtype dtype, void* stream);
fa_status fa_bwd_dq_convert(void* dq, const void* workspace, size_t workspace_bytes, int B, int H, int N, int d,
                            float scale, fa_dtype dtype, void* stream);

/*
 * The phases with options (opt as for fa_bwd_opt; NULL = defaults). With the
 * separate dQ pass (opt->dq_mode, or the library's choice): fa_bwd_preprocess_opt
 * does not zero the dQ accumulator; fa_bwd_main_opt computes dK and dV only and,
 * given dq, enqueues fa_bwd_dq_pass right after; fa_bwd_dq_pass is that pass on
 * its own: it reads D and LSE*log2e from the workspace (written by the
 * preprocess of the same call sequence) and writes dq [B,H,N,d] in full.
 * fa_bwd_opt is fa_bwd_preprocess_opt then fa_bwd_main_opt with dq given.
 */
fa_status fa_bwd_preprocess_opt(const void* o, const void* o_lo, const void* dO, const float* lse, void* workspace,
                                size_t workspace_bytes, int B, int H, int N, int d, int causal, fa_dtype dtype,
                                const fa_options* opt, void* stream);
fa_status fa_bwd_main_opt(const void* q, const void* k, const void* v, const void* dO, void* dk, void* dv, void* dq,
                          void* workspace, size_t workspace_bytes, int B, int H, int N, int d, float scale, int causal,
                          fa_dtype dtype, const fa_options* opt, void* stream);
fa_status fa_bwd_dq_pass(const void* q, const void* k, const void* v, const void* dO, void* dq, void* workspace,
                         size_t workspace_bytes, int B, int H, int N, int d, float scale, int causal, fa_dtype dtype,
                         const fa_options* opt, void* stream);

/* 1 if a backward with this head dimension, mask and options forms dQ with
 * the separate pass (then dq is bitwise reproducible), 0 if it accumulates it
 * (or the combination is not supported). opt may be NULL. */
int fa_bwd_uses_dq_pass(int d, int causal, const fa_options* opt);

/*
 * Paged decode attention: Mq new queries per sequence attend to the sequence's
 * cached keys and values, stored in fixed-size pages (the multi-query paged
 * attention kernel named on page "高级特性：探索PyTorch/XLA的Pallas内核和Flash
 * Attention实现", section "Pallas内核：自定义高效计算的关键"); per query the
 * online softmax of page "transformer模型详解（十）：FlashAttention优化技术",
 * section "Tiling 分块策略". The key range is cut into n_split splits handled
 * by different CTAs, each writing a partial (O_s, LSE_s) to the workspace, and a
 * second launch merges them: LSE = ln sum_s exp(LSE_s),
 * O = sum_s exp(LSE_s - LSE) O_s.
 *   q        [B, H, Mq, d] dtype: the queries at positions ctx_len[b] - Mq + i
 *   k_pages, v_pages  [Hkv, n_pages, page_size, d] dtype: the page pool
 *   page_table  DEVICE int32 [B, max_pages]: key j of sequence b lives in page
 *            page_table[b][j / page_size], row j % page_size. Entries for pages
 *            wholly past ctx_len[b] are never read; other entries outside
 *            [0, n_pages) read as zero keys/values.
 *   ctx_len  DEVICE int32 [B]: keys of sequence b (clamped to [0, max_pages *
 *            page_size]); values past it in the last page may hold anything.
 *   o        [B, H, Mq, d] dtype; lse [B, H, Mq] fp32 (a query that sees no
 *            key gets O = 0 and LSE = -inf).
 *   Query head h reads K/V head h / (H / Hkv). causal != 0: query i sees keys
 *   j <= ctx_len[b] - Mq + i; otherwise all ctx_len[b] keys.
 * Shapes: d in {64, 128, 256}; page_size a power of two in [16, 256]; H a
 * multiple of Hkv with (H / Hkv) * Mq <= 128; else FA_ERR_UNSUPPORTED.
 * n_split <= 0 lets the library choose (fa_decode_splits); at most 64 (32 for
 * d = 256; larger values are capped), and with one split the kernel writes o
 * and lse itself (no merge launch). workspace: device
 * memory of fa_decode_workspace_size(...) bytes for the same n_split,
 * 256-byte aligned. page_table and ctx_len must be 4-byte aligned, the rest
 * 16-byte aligned. One or two launches on `stream`.
 */
int fa_decode_splits(int B, int Hkv, int d, int page_size, int max_pages);
size_t fa_decode_workspace_size(int B, int H, int Hkv, int Mq, int d, int page_size, int max_pages, int n_split);
fa_status fa_decode(const void* q, const void* k_pages, const void* v_pages, const int* page_table, const int* ctx_len,
                    void* o, float* lse, void* workspace, size_t workspace_bytes, int B, int H, int Hkv, int Mq, int d,
                    int page_size, int n_pages, int max_pages, int n_split, float scale, int causal, fa_dtype dtype,
                    void* stream);

/*
 * Synchronises `stream`, then reads and clears the device status words of all
 * kernels. FA_OK if no kernel reported anything; FA_ERR_TIMEOUT if a bounded
 * wait expired; FA_ERR_DEVICE_FAULT for a failed device-side check;
 * FA_ERR_CUDA if the synchronisation itself failed.
 * If `info` is non-NULL it receives {code, where, block, count} of the first report:
 * code 1 = a bounded wait ran out, 2 = a failed index check; `where` names the
 * wait or check (1-20 forward, 31-39 decode, 41-59 backward, 90-99 self-tests);
 * `block` is the linear CTA index; `count` the number of reports.
 */
fa_status fa_device_status(void* stream, unsigned int info[4]);

/* Static, human-readable name of a status code. */
const char* fa_status_string(fa_status s);

/*
 * Upper bound, in nanoseconds, of every device-side wait (default 4e9).
 * Takes effect for launches after the call; 0 restores the default.
 */
void fa_set_wait_timeout_ns(unsigned long long ns);

/* ABI version (major*100 + minor). */
int fa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FA_H_ */
