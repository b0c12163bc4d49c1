// Descriptor self-test: one CTA computes D[128 x n] = A[128 x k] * B[n x k]^T with
// tcgen05.mma, using exactly the operand forms the attention kernels use
// (K-major and MN-major operands in 128-byte-swizzled shared memory filled by
// TMA, and an A operand held in tensor memory). Tests compare it with a CPU
// matrix product, which checks the hand-encoded shared-memory descriptors, the
// instruction descriptor, the TMEM data-path layout and the 16-bit packing of
// TMEM operands independently of any attention arithmetic.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/fa.h"
#include "../../include/fa_selftest.h"
#include "common.cuh"
#include "fa_bwd_order.cuh"
#include "launch.h"

namespace fa {
namespace {

struct STParams {
  CUtensorMap tm_a, tm_b;
  const uint32_t* a_glob;  // for a_mode 2: a[128][k] as 16-bit pairs
  float* d;
  int n, k, a_mode, b_mode;
  unsigned long long timeout_ns;
};

constexpr int ST_SMEM = 1024 + 32768 + 65536 + 64;

template <bool BF16>
__global__ void __launch_bounds__(128, 1) fa_selftest_kernel(const __grid_constant__ STParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sA = smem_u32(smem);
  const uint32_t sB = sA + 32768;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + 32768 + 65536);
  const uint32_t b_ld = smem_u32(&bars[0]), b_mma = smem_u32(&bars[1]);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(&bars[2]);
  volatile uint32_t* abort_flag = tmem_slot + 1;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n = p.n, k = p.k;

  if (threadIdx.x == 0) {
    mbar_init(b_ld, 1);
    mbar_init(b_mma, 1);
    *abort_flag = 0u;
    mbar_fence_init();
    fence_proxy_async_smem();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;

  if (threadIdx.x == 0) {
    uint32_t bytes = static_cast<uint32_t>(n * k * 2);
    if (p.a_mode < 2) bytes += 128u * k * 2;
    mbar_arrive_expect_tx(b_ld, bytes);
    if (p.a_mode == 0)
      for (int c = 0; c < k / 64; ++c) tma_load_2d(sA + c * 16384, &p.tm_a, b_ld, c * 64, 0);
    else if (p.a_mode == 1)
      for (int c = 0; c < 2; ++c) tma_load_2d(sA + c * (k * 128), &p.tm_a, b_ld, c * 64, 0);
    if (p.b_mode == 0)
      for (int c = 0; c < k / 64; ++c) tma_load_2d(sB + c * (n * 128), &p.tm_b, b_ld, c * 64, 0);
    else
      for (int c = 0; c < n / 64; ++c) tma_load_2d(sB + c * (k * 128), &p.tm_b, b_ld, c * 64, 0);
  }
  if (p.a_mode == 2) {
    // row threadIdx.x of A -> TMEM lane threadIdx.x, columns 256 .. 256 + k/2 (two 16-bit values per column)
    const uint32_t* row = p.a_glob + static_cast<size_t>(threadIdx.x) * (k / 2);
    for (int c = 0; c < k / 64; ++c) {
      uint32_t u[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) u[i] = row[32 * c + i];
      tmem_st32(tmem + lane_off + 256 + 32 * c, u);
    }
    tmem_st_wait();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  if (threadIdx.x == 0) {
    if (wait_bar(b_ld, 0, p.timeout_ns, abort_flag, 1)) {
      tc_fence_after();
      const uint32_t idesc = make_idesc(128, n, BF16, p.a_mode == 1, p.b_mode == 1);
      for (int kk = 0; kk < k / 16; ++kk) {
        const uint64_t bdesc = (p.b_mode == 0)
                                   ? make_sdesc(sB + (kk >> 2) * (n * 128) + (kk & 3) * 32, 16, 1024)
                                   : make_sdesc(sB + kk * 2048, k * 128, 1024);
        if (p.a_mode == 2) {
          mma_ts(tmem, tmem + 256 + kk * 8, bdesc, idesc, kk > 0 ? 1u : 0u);
        } else {
          const uint64_t adesc = (p.a_mode == 0) ? make_sdesc(sA + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024)
                                                 : make_sdesc(sA + kk * 2048, k * 128, 1024);
          mma_ss(tmem, adesc, bdesc, idesc, kk > 0 ? 1u : 0u);
        }
      }
    }
    mma_commit(b_mma);
  }
  __syncwarp();
  const bool ok = __all_sync(0xffffffffu, wait_bar(b_mma, 0, p.timeout_ns, abort_flag, 2));
  if (ok) {
    tc_fence_after();
    for (int c = 0; c < n / 32; ++c) {
      uint32_t u[32];
      tmem_ld32(tmem + lane_off + 32 * c, u);
      float* out = p.d + static_cast<size_t>(warp * 32 + lane) * n + 32 * c;
#pragma unroll
      for (int i = 0; i < 32; ++i) out[i] = __uint_as_float(u[i]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

bool st_map(CUtensorMap* m, const void* base, int rows, int cols, bool bf16, int box_rows) {
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess)
    return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 2};
  cuuint32_t box[2] = {64u, static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[2] = {1u, 1u};
  return reinterpret_cast<EncodeTiledFn>(fn)(
             m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(base),
             dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace
}  // namespace fa

extern "C" fa_status fa_selftest_gemm(const void* a, const void* b, float* d, int n, int k, int a_mode, int b_mode,
                                      fa_dtype dtype, void* stream) {
  using namespace fa;
  if (!a || !b || !d) return FA_ERR_INVALID_ARG;
  if (dtype != FA_F16 && dtype != FA_BF16) return FA_ERR_INVALID_ARG;
  if (!(n == 64 || n == 128 || n == 256) || !(k == 64 || k == 128)) return FA_ERR_UNSUPPORTED;
  if (a_mode < 0 || a_mode > 2 || b_mode < 0 || b_mode > 1) return FA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(a) | reinterpret_cast<uintptr_t>(b) | reinterpret_cast<uintptr_t>(d)) & 15u)
    return FA_ERR_ALIGNMENT;
  int dev = 0, major = 0, minor = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_CUDA;
  cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
  cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
  if (major != 10 || minor != 3) return FA_ERR_UNSUPPORTED;
  const bool bf16 = dtype == FA_BF16;
  STParams p{};
  // A: mode 0 -> [128][k] (box 128 rows); mode 1 -> [k][128] (box k rows); mode 2 -> read by threads
  if (a_mode == 0 && !st_map(&p.tm_a, a, 128, k, bf16, 128)) return FA_ERR_CUDA;
  if (a_mode == 1 && !st_map(&p.tm_a, a, k, 128, bf16, k)) return FA_ERR_CUDA;
  if (a_mode == 2) p.tm_a = CUtensorMap{};
  if (b_mode == 0 && !st_map(&p.tm_b, b, n, k, bf16, n)) return FA_ERR_CUDA;
  if (b_mode == 1 && !st_map(&p.tm_b, b, k, n, bf16, k)) return FA_ERR_CUDA;
  p.a_glob = static_cast<const uint32_t*>(a);
  p.d = d;
  p.n = n;
  p.k = k;
  p.a_mode = a_mode;
  p.b_mode = b_mode;
  p.timeout_ns = 2000000000ull;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (bf16) {
    if (cudaFuncSetAttribute(fa_selftest_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, ST_SMEM) !=
        cudaSuccess)
      return FA_ERR_CUDA;
    fa_selftest_kernel<true><<<1, 128, ST_SMEM, s>>>(p);
  } else {
    if (cudaFuncSetAttribute(fa_selftest_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, ST_SMEM) !=
        cudaSuccess)
      return FA_ERR_CUDA;
    fa_selftest_kernel<false><<<1, 128, ST_SMEM, s>>>(p);
  }
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

// ---------------------------------------------------------------- MMA issue-rate microbenchmark
// One CTA per SM issues `reps` x 8 back-to-back tcgen05.mma (M = 128, K = 16, bf16 -> fp32) of one
// shape from a single thread, rotating over n_acc independent accumulators (consecutive
// instructions then do not depend on each other when n_acc > 1), and records the clock64 cycles
// from the first issue to the completion of the last (tcgen05.commit + mbarrier). Operands are zeroed shared memory (K-major, 128-byte
// swizzle) or zeroed TMEM columns; only the timing is of interest.
namespace fa {
namespace {
constexpr int MR_SMEM = 1024 + 16384 + 32768 + 128;

__global__ void __launch_bounds__(128, 1) fa_mma_rate_kernel(int n, int a_tmem, int n_acc, int tmem_mode, int reps,
                                                            unsigned long long* out, unsigned long long timeout_ns) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sA = smem_u32(smem), sB = sA + 16384;
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + 16384 + 32768);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + 1);
  volatile uint32_t* abort_flag = tmem_slot + 1;
  const int warp = threadIdx.x >> 5;
  for (int i = threadIdx.x; i < (16384 + 32768) / 16; i += 128) reinterpret_cast<uint4*>(smem)[i] = make_uint4(0, 0, 0, 0);
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(bar), 1);
    mbar_init(smem_u32(bar + 2), 1);
    *abort_flag = 0u;
    mbar_fence_init();
  }
  fence_proxy_async_smem();
  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_ld_base = *tmem_slot;
  const uint32_t tmem = tmem_ld_base;
  if (tmem_mode == 2 && tmem != 0u) report_status(FA_DEV_BAD_INDEX, 99);
  {
    uint32_t z[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) z[i] = 0u;
    tmem_st32(tmem + (static_cast<uint32_t>(warp * 32) << 16) + 480, z);
    tmem_st_wait();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // tmem_mode 3: threads 0 and 32 both issue, each into its own accumulator columns.
  if (threadIdx.x == 0 || (tmem_mode == 3 && threadIdx.x == 32)) {
    // tmem_mode 0: base address as loaded from shared memory; 1: broadcast with a shuffle;
    // 2: the constant 0 (a CTA that owns all 512 columns always gets column 0, lane 0).
    const uint32_t tmem = tmem_mode == 2 ? 0u : (tmem_mode == 1 ? __shfl_sync(1u, tmem_ld_base, 0) : tmem_ld_base);
    const uint32_t idesc = make_idesc(128, n, true, false, false);
    const uint64_t da = make_sdesc(sA, 16, 1024), db = make_sdesc(sB, 16, 1024);
    const long long t0 = clock64();
    for (int r = 0; r < reps; ++r) {
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const uint64_t off = static_cast<uint64_t>((kk & 3) * 32) >> 4;
        const uint32_t d = tmem + static_cast<uint32_t>((kk % n_acc) * n) + (threadIdx.x == 32 ? 256u : 0u);
        if (a_tmem)
          mma_ts(d, tmem + 480 + (kk & 3) * 8, db + off, idesc, 1u);
        else
          mma_ss(d, da + off, db + off, idesc, 1u);
      }
    }
    const uint32_t mybar = smem_u32(threadIdx.x == 32 ? bar + 2 : bar);
    mma_commit(mybar);
    wait_bar(mybar, 0, timeout_ns, abort_flag, 1);
    if (threadIdx.x == 0) out[blockIdx.x] = static_cast<unsigned long long>(clock64() - t0);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}
}  // namespace
}  // namespace fa

extern "C" fa_status fa_selftest_mma_rate(int n, int a_tmem, int n_acc, int reps, int blocks,
                                          unsigned long long* cycles, void* stream) {
  const int tmem_mode = (n_acc >> 4) & 3;  // test-only: bits 4-5 select how the TMEM base is obtained
  n_acc &= 15;
  using namespace fa;
  if (!cycles) return FA_ERR_INVALID_ARG;
  if (!(n == 64 || n == 128 || n == 256) || reps < 1 || reps > (1 << 20) || blocks < 1 || blocks > 4096)
    return FA_ERR_UNSUPPORTED;
  if (!(n_acc == 1 || n_acc == 2 || n_acc == 4) || n * n_acc > (a_tmem ? 480 : 512)) return FA_ERR_UNSUPPORTED;
  int dev = 0, major = 0, minor = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_CUDA;
  cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
  cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
  if (major != 10 || minor != 3) return FA_ERR_UNSUPPORTED;
  if (cudaFuncSetAttribute(fa_mma_rate_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, MR_SMEM) != cudaSuccess)
    return FA_ERR_CUDA;
  fa_mma_rate_kernel<<<blocks, 128, MR_SMEM, static_cast<cudaStream_t>(stream)>>>(n, a_tmem ? 1 : 0, n_acc, tmem_mode, reps, cycles,
                                                                                 2000000000ull);
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

// ---------------------------------------------------------------- MMA operand-pattern microbenchmark
// Like the issue-rate test, but with the operand pattern of the attention kernels: random 16-bit
// data, two distinct B tiles (and two distinct A tiles) used in turn, whole K = 128 products (8
// instructions, the first overwriting the accumulator), K-major or MN-major operands, A from shared
// memory or from TMEM, and 1 to 4 issuing threads (lane 0 of warps 0..3), each with its own
// accumulators. Modes:
//   0  one K = 128 product after another, each into the next of the issuer's accumulators (all SS,
//      or all TS with a_tmem);
//   1  the forward's pattern: an SS product (S = Q K^T) and a TS product (O += P V) in turn, into two
//      accumulators (needs a_tmem for the TS operand);
//   2  two SS products interleaved instruction by instruction into two accumulators (two
//      independent accumulation chains in flight from one thread).
// An SS instruction reads 128 x 16 (A) + n x 16 (B) 16-bit elements from shared memory, a TS
// instruction only the B part.
namespace fa {
namespace {
constexpr int MP_A_TILE = 2 * 16384;   // 128 rows x 128 K elements (two 64-wide chunks)
constexpr int MP_B_TILE = 2 * 32768;   // up to 256 rows x 128 K elements
constexpr int MP_SMEM = 1024 + 2 * MP_A_TILE + 2 * MP_B_TILE + 128;

__global__ void __launch_bounds__(128, 1) fa_mma_pattern_kernel(int n, int a_tmem, int a_mn, int b_mn, int issuers,
                                                                int mode, int n_buf, int reps,
                                                                unsigned long long* out,
                                                                unsigned long long timeout_ns) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sA = smem_u32(smem), sB = sA + 2 * MP_A_TILE;
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + 2 * MP_A_TILE + 2 * MP_B_TILE);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + 4);
  volatile uint32_t* abort_flag = tmem_slot + 1;
  const int warp = threadIdx.x >> 5;
  // random bf16 in about (-1, 1): a hash of the element index, exponent fixed at 2^-1
  uint32_t* w = reinterpret_cast<uint32_t*>(smem);
  for (int i = threadIdx.x; i < (2 * MP_A_TILE + 2 * MP_B_TILE) / 4; i += 128) {
    uint32_t h = static_cast<uint32_t>(i) * 2654435761u + 0x9E3779B9u * static_cast<uint32_t>(blockIdx.x);
    h ^= h >> 15;
    h *= 2246822519u;
    h ^= h >> 13;
    w[i] = (h & 0x807F807Fu) | 0x3F003F00u;
  }
  if (threadIdx.x == 0) {
    for (int i = 0; i < 4; ++i) mbar_init(smem_u32(bar + i), 1);
    *abort_flag = 0u;
    mbar_fence_init();
  }
  fence_proxy_async_smem();
  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t a_col = 448;  // A operand in TMEM: 128 lanes x 128 K elements as 64 packed columns
  if (a_tmem) {
    uint32_t z[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) z[i] = 0x3F003F00u ^ ((threadIdx.x * 7u + i * 13u) & 0x007F007Fu);
    tmem_st32(tmem + (static_cast<uint32_t>(warp * 32) << 16) + a_col, z);
    tmem_st32(tmem + (static_cast<uint32_t>(warp * 32) << 16) + a_col + 32, z);
    tmem_st_wait();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const int lane = threadIdx.x & 31;
  if (warp < issuers && lane == 0) {
    const uint32_t idesc = make_idesc(128, n, true, a_mn != 0, b_mn != 0);
    const uint32_t idesc_ts = make_idesc(128, n, true, false, b_mn != 0);
    // K-major: rows of 128 bytes (64 K elements), 8-row groups 1024 bytes apart, a K step of 16 is
    // 32 bytes inside the row, the second 64-wide K chunk a whole chunk further on.
    // MN-major: rows are K indices of 64 M/N elements; LBO = distance between 64-wide M/N chunks,
    // a K step of 16 is 16 rows (2048 bytes).
    const uint32_t a_chunk = 128 * 128, b_chunk = static_cast<uint32_t>(n) * 128;
    const uint64_t da = a_mn ? make_sdesc(sA, 128 * 128, 1024) : make_sdesc(sA, 16, 1024);
    const uint64_t db = b_mn ? make_sdesc(sB, 128 * 128, 1024) : make_sdesc(sB, 16, 1024);
    const uint32_t acc0 = tmem + static_cast<uint32_t>(warp * n_buf * n);
    auto ss = [&](uint32_t d, uint32_t tile, int kk) {
      const uint32_t oa = a_mn ? kk * 2048u : (kk >> 2) * a_chunk + (kk & 3) * 32u;
      const uint32_t ob = b_mn ? kk * 2048u : (kk >> 2) * b_chunk + (kk & 3) * 32u;
      mma_ss(d, da + (static_cast<uint64_t>(tile * MP_A_TILE + oa) >> 4),
             db + (static_cast<uint64_t>(tile * MP_B_TILE + ob) >> 4), idesc, kk > 0 ? 1u : 0u);
    };
    auto ts = [&](uint32_t d, uint32_t tile, int kk) {
      const uint32_t ob = b_mn ? kk * 2048u : (kk >> 2) * b_chunk + (kk & 3) * 32u;
      mma_ts(d, tmem + a_col + kk * 8, db + (static_cast<uint64_t>(tile * MP_B_TILE + ob) >> 4), idesc_ts,
             kk > 0 ? 1u : 0u);
    };
    const long long t0 = clock64();
    for (int r = 0; r < reps; ++r) {
      const uint32_t tile = static_cast<uint32_t>(r & 1);
      if (mode == 0) {
        const uint32_t d = acc0 + static_cast<uint32_t>((r % n_buf) * n);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          if (a_tmem)
            ts(d, tile, kk);
          else
            ss(d, tile, kk);
        }
      } else if (mode == 1) {
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          if (r & 1)
            ts(acc0 + n, tile, kk);
          else
            ss(acc0, tile, kk);
        }
      } else {
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          ss(acc0, tile, kk);
          ss(acc0 + n, tile ^ 1u, kk);
        }
      }
    }
    const uint32_t mybar = smem_u32(bar + warp);
    mma_commit(mybar);
    wait_bar(mybar, 0, timeout_ns, abort_flag, 98);
    out[blockIdx.x * 4 + warp] = static_cast<unsigned long long>(clock64() - t0);
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}
}  // namespace
}  // namespace fa

extern "C" fa_status fa_selftest_mma_pattern(int n, int a_tmem, int a_mn, int b_mn, int issuers, int mode, int reps,
                                             int blocks, unsigned long long* cycles, void* stream) {
  using namespace fa;
  if (!cycles) return FA_ERR_INVALID_ARG;
  if (!(n == 64 || n == 128 || n == 256) || issuers < 1 || issuers > 4 || mode < 0 || mode > 2 || reps < 1 ||
      reps > (1 << 20) || blocks < 1 || blocks > 4096)
    return FA_ERR_UNSUPPORTED;
  if (a_tmem && a_mn) return FA_ERR_UNSUPPORTED;  // a TMEM operand has no major-ness choice
  if (mode == 1 && !a_tmem) return FA_ERR_UNSUPPORTED;  // the TS products need the TMEM operand
  // accumulators per issuer: mode 0 two where they fit (else one), modes 1 and 2 exactly two; all of
  // them next to the TMEM A operand (columns 448..511) when there is one
  const int room = a_tmem ? 448 : 512;
  int n_buf = mode == 0 ? ((issuers * 2 * n <= room) ? 2 : 1) : 2;
  if (issuers * n_buf * n > room) return FA_ERR_UNSUPPORTED;
  int dev = 0, major = 0, minor = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_CUDA;
  cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
  cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
  if (major != 10 || minor != 3) return FA_ERR_UNSUPPORTED;
  if (cudaFuncSetAttribute(fa_mma_pattern_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, MP_SMEM) !=
      cudaSuccess)
    return FA_ERR_CUDA;
  fa_mma_pattern_kernel<<<blocks, 128, MP_SMEM, static_cast<cudaStream_t>(stream)>>>(
      n, a_tmem ? 1 : 0, a_mn ? 1 : 0, b_mn ? 1 : 0, issuers, mode, n_buf, reps, cycles, 2000000000ull);
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

// A wait that nothing completes: one thread waits on an mbarrier phase that no thread or copy will
// ever finish. The bounded wait gives up after timeout_ns, records FA_DEV_TIMEOUT (where-code 90) in
// this translation unit's status word and the kernel returns: nothing else is in flight, so the
// context stays usable. This is how every kernel of the library reports a wait that ran out.
namespace fa {
namespace {
constexpr uint32_t WT_WHERE = 90;
__global__ void __launch_bounds__(32, 1) fa_wait_timeout_kernel(unsigned long long timeout_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ uint32_t abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0u;
    mbar_fence_init();
  }
  __syncwarp();
  if (threadIdx.x == 0) wait_bar(smem_u32(&bar), 0, timeout_ns, &abort_flag, WT_WHERE);
  __syncwarp();
}
}  // namespace

cudaError_t read_clear_status_selftest(DevStatusHost* out, cudaStream_t s) {
  DevStatus zero{0, 0, 0, 0};
  cudaError_t e = cudaMemcpyFromSymbolAsync(out, g_status, sizeof(DevStatus), 0, cudaMemcpyDeviceToHost, s);
  if (e != cudaSuccess) return e;
  e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return e;
  if (out->code != 0 || out->count != 0)
    e = cudaMemcpyToSymbolAsync(g_status, &zero, sizeof(DevStatus), 0, cudaMemcpyHostToDevice, s);
  if (e != cudaSuccess) return e;
  return cudaStreamSynchronize(s);
}
}  // namespace fa

extern "C" fa_status fa_selftest_wait_timeout(unsigned long long timeout_ns, void* stream) {
  if (timeout_ns < 1000ull || timeout_ns > 1000000000ull) return FA_ERR_INVALID_ARG;  // 1 us .. 1 s
  int dev = 0, major = 0, minor = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_CUDA;
  cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
  cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
  if (major != 10 || minor != 3) return FA_ERR_UNSUPPORTED;
  fa::fa_wait_timeout_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(timeout_ns);
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

// Exponential-unit rate microbenchmark: every thread runs 8 independent chains of `reps` dependent
// ex2.approx.f32 (x <- 2^x - 1.5 keeps x in [-1, 0]), so the special-function units, not latency,
// set the pace once enough warps are resident. The sum of the chains goes to sink[block] so that
// nothing is optimised away. Timed by the caller (events around the launch).
namespace fa {
namespace {
__global__ void __launch_bounds__(512) fa_ex2_rate_kernel(int reps, float* sink) {
  float x[8];
#pragma unroll
  for (int c = 0; c < 8; ++c) x[c] = -0.125f * static_cast<float>(c + 1) - 1e-6f * static_cast<float>(threadIdx.x);
#pragma unroll 1
  for (int r = 0; r < reps; ++r) {
#pragma unroll
    for (int c = 0; c < 8; ++c) x[c] = ex2_approx(x[c]) - 1.5f;
  }
  float s = 0.f;
#pragma unroll
  for (int c = 0; c < 8; ++c) s += x[c];
  s += __shfl_xor_sync(0xffffffffu, s, 16);
  if ((threadIdx.x & 31) == 0) atomicAdd(sink + blockIdx.x, s);
}
}  // namespace
}  // namespace fa

extern "C" fa_status fa_selftest_ex2_rate(int reps, int blocks, float* sink, void* stream) {
  if (!sink) return FA_ERR_INVALID_ARG;
  if (reps < 1 || reps > (1 << 20) || blocks < 1 || blocks > 65535) return FA_ERR_UNSUPPORTED;
  int dev = 0, major = 0, minor = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_CUDA;
  cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
  cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
  if (major != 10 || minor != 3) return FA_ERR_UNSUPPORTED;
  fa::fa_ex2_rate_kernel<<<blocks, 512, 0, static_cast<cudaStream_t>(stream)>>>(reps, sink);
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

namespace fa {
namespace {
__global__ void fa_block_order_kernel(int heads, int nkb, long long head_bytes, int* out) {
  const long long n = static_cast<long long>(heads) * nkb;
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int x = static_cast<int>(i % heads), y = static_cast<int>(i / heads);
    int bh, kb;
    bwd_block_order(x, y, heads, nkb, head_bytes, bh, kb);
    out[i] = bh * nkb + kb;
  }
}
}  // namespace
}  // namespace fa

extern "C" fa_status fa_selftest_block_order(int heads, int nkb, long long head_bytes, int* out, void* stream) {
  if (!out) return FA_ERR_INVALID_ARG;
  if (heads < 1 || nkb < 1 || head_bytes < 1 || static_cast<long long>(heads) * nkb >= (1ll << 31))
    return FA_ERR_UNSUPPORTED;
  fa::fa_block_order_kernel<<<256, 256, 0, static_cast<cudaStream_t>(stream)>>>(heads, nkb, head_bytes, out);
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

namespace fa {
namespace {
__global__ void __launch_bounds__(512) fa_copy_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst,
                                                      size_t n) {
  const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
  size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  for (; i + 3 * stride < n; i += 4 * stride) {  // four loads in flight per thread
    const uint4 a = src[i], b = src[i + stride], c = src[i + 2 * stride], d = src[i + 3 * stride];
    dst[i] = a;
    dst[i + stride] = b;
    dst[i + 2 * stride] = c;
    dst[i + 3 * stride] = d;
  }
  for (; i < n; i += stride) dst[i] = src[i];
}
}  // namespace
}  // namespace fa

// The address the GPU uses for p: device (or managed) memory as it is, pinned host memory through its
// mapping; anything else (pageable host memory) is refused.
static bool fa_gpu_address(const void* p, const void** out) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  if (a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged) {
    *out = p;
    return true;
  }
  if (a.type == cudaMemoryTypeHost && a.devicePointer != nullptr) {
    *out = a.devicePointer;
    return true;
  }
  return false;
}

extern "C" fa_status fa_selftest_copy(const void* src, void* dst, size_t bytes, int blocks, void* stream) {
  if (!src || !dst) return FA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(src) | reinterpret_cast<uintptr_t>(dst) | bytes) & 15) return FA_ERR_ALIGNMENT;
  if (blocks < 1 || blocks > 65535) return FA_ERR_UNSUPPORTED;
  const void *gs = nullptr, *gd = nullptr;
  if (!fa_gpu_address(src, &gs) || !fa_gpu_address(dst, &gd)) return FA_ERR_INVALID_ARG;
  fa::fa_copy_kernel<<<blocks, 512, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<const uint4*>(gs), static_cast<uint4*>(const_cast<void*>(gd)), bytes / 16);
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}
