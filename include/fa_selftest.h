/*
 * fa_selftest.h — tensor-core building-block self-test exported by libfa.so.
 *
 * Not part of the attention method: the pages have no counterpart. It checks,
 * in isolation, the operand forms the attention kernels feed to tcgen05.mma,
 * so that a descriptor or layout mistake shows up as a wrong matrix product
 * rather than as a wrong attention result.
 *
 * Computes, with one CTA on the current device,
 *     d[i][j] = sum_t A[i][t] * B[j][t]      (i < 128, j < n, t < k), fp32
 * from 16-bit inputs of type `dtype`. Storage of the operands in DEVICE memory:
 *   a_mode 0: a = A stored [128][k] (row-major, k contiguous) -> smem, K-major
 *   a_mode 1: a = A stored [k][128] (A transposed)            -> smem, MN-major
 *   a_mode 2: a = A stored [128][k]                           -> tensor memory
 *   b_mode 0: b = B stored [n][k]                             -> smem, K-major
 *   b_mode 1: b = B stored [k][n] (B transposed)              -> smem, MN-major
 *   d: fp32 [128][n] row-major, written in full.
 * n in {64, 128, 256}, k in {64, 128}; pointers 16-byte aligned.
 * Returns FA_OK after enqueuing on `stream` (a cudaStream_t as void*), or an
 * argument / device error from fa.h without launching.
 */
#ifndef FA_SELFTEST_H_
#define FA_SELFTEST_H_

#include "fa.h"

#ifdef __cplusplus
extern "C" {
#endif

fa_status fa_selftest_gemm(const void* a, const void* b, float* d, int n, int k, int a_mode, int b_mode,
                           fa_dtype dtype, void* stream);

/*
 * Tensor-core rate microbenchmark: `blocks` CTAs (one per SM when blocks is
 * the SM count) each issue reps x 8 back-to-back tcgen05.mma of shape
 * M = 128, N = n, K = 16 (bf16 -> fp32) from one thread, A from shared memory
 * (a_tmem = 0) or from tensor memory (a_tmem = 1), B from shared memory,
 * cycling over n_acc in {1, 2, 4} independent accumulators (n * n_acc <= 512,
 * <= 480 with a_tmem), and
 * write the clock64 cycles from first issue to completion to cycles[block]
 * (DEVICE pointer, `blocks` entries). Cycles / (8 reps) is the sustained cost
 * of one instruction of that shape; 2*128*n*16 / that is FLOP/clock/SM.
 * n in {64, 128, 256}; 1 <= reps <= 2^20; 1 <= blocks <= 4096.
 */
fa_status fa_selftest_mma_rate(int n, int a_tmem, int n_acc, int reps, int blocks, unsigned long long* cycles,
                               void* stream);

/*
 * Tensor-core operand-pattern microbenchmark: like fa_selftest_mma_rate, but
 * with the operand pattern of the attention kernels. Each CTA fills its shared
 * memory with random 16-bit values; `issuers` threads (1 to 4, lane 0 of warps
 * 0..3, each with its own accumulators) each issue `reps` products of K = 128
 * (8 tcgen05.mma of M = 128, N = n, K = 16, the first of each overwriting its
 * accumulator), alternating between two distinct A tiles and two distinct B
 * tiles. a_tmem = 1 takes A from tensor memory (then a_mn must be 0); a_mn /
 * b_mn = 1 lay A / B out MN-major instead of K-major (128-byte swizzle either
 * way). mode 0: product after product (all SS, or all TS with a_tmem); mode
 * 1: an SS and a TS product in turn, as the forward issues S = Q K^T and
 * O += P V (needs a_tmem); mode 2: two SS products interleaved instruction by
 * instruction into two accumulators (each rep then holds 16 instructions).
 * cycles: DEVICE array of 4 * blocks entries; entry 4*block + i receives
 * issuer i's clock64 cycles from its first issue to the completion of its last
 * instruction. n in {64, 128, 256}; the issuers' accumulators must fit in
 * tensor memory (else FA_ERR_UNSUPPORTED).
 */
fa_status fa_selftest_mma_pattern(int n, int a_tmem, int a_mn, int b_mn, int issuers, int mode, int reps, int blocks,
                                  unsigned long long* cycles, void* stream);

/*
 * Failure-detection self-test: one kernel waits (bounded, like every wait in
 * the library) on an mbarrier phase that nothing completes. After timeout_ns
 * (1e3 .. 1e9, else FA_ERR_INVALID_ARG) it records a timeout in the device
 * status word and returns; fa_device_status then reports FA_ERR_TIMEOUT with
 * info[1] = 90, and the context stays usable. Nothing traps or hangs.
 */
fa_status fa_selftest_wait_timeout(unsigned long long timeout_ns, void* stream);

/*
 * Exponential-unit rate microbenchmark (the secondary roofline of the softmax):
 * `blocks` CTAs of 512 threads each run 8 independent chains of `reps`
 * dependent ex2.approx.f32, i.e. blocks * 512 * 8 * reps exponentials; the
 * caller times the launch. sink: DEVICE float[blocks], zeroed by the caller
 * (receives the chains' sums). 1 <= reps <= 2^20, 1 <= blocks <= 65535.
 */
fa_status fa_selftest_ex2_rate(int reps, int blocks, float* sink, void* stream);

/*
 * The backward main kernels' work order: for every launch index
 * i = x + heads * y of a grid of heads x nkb CTAs, out[i] = bh * nkb + kb, the
 * K/V head and 128-key block that CTA (x, y) works on, as the kernels compute
 * it (heads taken in groups whose shared rows, head_bytes each, fit in about
 * 64 MB, longest blocks first within a group). out: DEVICE int[heads * nkb].
 * 1 <= heads, 1 <= nkb, heads * nkb < 2^31, head_bytes >= 1.
 */
fa_status fa_selftest_block_order(int heads, int nkb, long long head_bytes, int* out, void* stream);

/*
 * Copy-rate microbenchmark of the GPU's own loads and stores: `blocks` CTAs of
 * 512 threads copy `bytes` from src to dst in 16-byte vectors (grid-stride),
 * where src and dst may be device memory or pinned host memory (which the
 * GPU addresses directly, through the mapping CUDA reports for it); the
 * caller times the launch. Memory that CUDA reports neither as device
 * memory nor as mapped pinned host memory is refused (FA_ERR_INVALID_ARG). src, dst: 16-byte aligned, bytes a multiple of 16,
 * 1 <= blocks <= 65535.
 */
fa_status fa_selftest_copy(const void* src, void* dst, size_t bytes, int blocks, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* FA_SELFTEST_H_ */
