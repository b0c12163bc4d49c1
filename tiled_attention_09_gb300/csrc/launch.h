// Host-side interface between the C ABI (fa_api.cu) and the kernel translation units.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>

namespace fa {

// Raises a kernel's dynamic shared-memory limit once per device: cudaFuncSetAttribute costs host
// time on every call, and decode steps are short enough for that to show.
inline cudaError_t smem_attr_once(const void* kern, int bytes, std::atomic<unsigned long long>& done) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = dev < 64 ? (1ull << dev) : 0ull;
  if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_acq_rel);
  return e;
}

// Plain stream-ordered launch, returning the launch error.
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                          Args&&... args) {
  kern<<<grid, block, smem, stream>>>(static_cast<Args&&>(args)...);
  return cudaGetLastError();
}

struct DevStatusHost {
  uint32_t code, where, block, count;
};

// 3-D tensor maps over [heads][N][d] (heads = B*H for Q, dO, O; B*Hkv for K, V, dK, dV),
// box {64 elements, box_rows rows, 1}, 128-byte swizzle.
struct FwdArgs {
  CUtensorMap tm_q, tm_k, tm_v;  // box rows 128
  void* o;     // [B*H*N, d] output, in the input dtype or (o_f32) fp32
  float* lse;
  void* o_lo;  // optional rounding residual of O (nullptr: not written)
  const int* kv_len;  // optional [B] key counts (key-padding mask)
  int kv_splits;      // CTAs per query block's key range (1: no split)
  int tiles_per_item; // query tiles per work item without a split: 0 = the kernel's two (d <= 128), or 1
  float* part_o;      // kv_splits > 1: [kv_splits][B*H*N][d] fp32 partial outputs
  float* part_lse;    // kv_splits > 1: [kv_splits][B*H*N] their LSEs
  int B, H, Hkv, N, d;
  bool o_f32;
  float scale;
  bool causal, bf16;
  uint64_t timeout_ns;
  cudaStream_t stream;
};

struct BwdArgs {
  CUtensorMap tm_q, tm_k, tm_v, tm_do;  // q, dO: box rows = query tile; k, v: box rows 128
  CUtensorMap tm_dk, tm_dv;             // box rows 128
  const void* o;      // dtype, or fp32 when o_f32
  const void* o_lo;  // optional rounding residual of O (nullptr: D from o alone)
  const int* kv_len;  // optional [B] key counts (key-padding mask)
  const void* dO;
  const float* lse;
  void* dq;
  void* dk;
  void* dv;
  float* ws_D;      // [B*H*Npad]: row (bh, r) at bh * Npad + r, Npad = N rounded up to 128
  float* ws_lse2;   // [B*H*Npad]  lse * log2(e)
  float* ws_dqacc;  // [B*H*Npad*d]
  int B, H, Hkv, N, d;
  int Npad;  // N rounded up to 128: the per-head row stride of the workspace arrays
  bool dq_pass;  // dQ by the separate query-major pass (no accumulator) instead of accumulation
  bool o_f32;
  float scale;
  bool causal, bf16;
  uint64_t timeout_ns;
  cudaStream_t stream;
};

// Paged decode: q [B*H*Mq, d] (2-D map, box rows 128); k, v pages [Hkv][n_pages*page_size][d]
// (3-D maps, box rows min(page_size, 128)); partial results in the workspace.
struct DecArgs {
  CUtensorMap tm_q, tm_k, tm_v;
  const int* page_table;  // [B][max_pages]
  const int* ctx_len;     // [B]
  float* ws_o;            // [n_split][B*H*Mq][d]
  float* ws_lse;          // [n_split][B*H*Mq]
  void* o;                // [B*H*Mq, d] dtype
  float* lse;             // [B*H*Mq]
  int B, H, Hkv, Mq, d;
  int ps_log2, max_pages, n_pages;
  int tiles_per_split, n_split;
  float scale;
  bool causal, bf16;
  uint64_t timeout_ns;
  cudaStream_t stream;
};

// Query-tile height of the backward main kernel for head dimension d (0 = unsupported).
inline int bwd_query_tile(int d) { return (d == 64 || d == 128 || d == 256) ? 64 : 0; }

cudaError_t launch_fwd(const FwdArgs& a);
cudaError_t launch_bwd_preprocess(const BwdArgs& a);
cudaError_t launch_bwd_main(const BwdArgs& a);
cudaError_t launch_bwd_dq_convert(const BwdArgs& a);
cudaError_t launch_bwd_dq_pass(const BwdArgs& a);

cudaError_t read_clear_status_fwd(DevStatusHost* out, cudaStream_t s);
cudaError_t read_clear_status_bwd(DevStatusHost* out, cudaStream_t s);
cudaError_t launch_decode(const DecArgs& a);
cudaError_t read_clear_status_decode(DevStatusHost* out, cudaStream_t s);
cudaError_t read_clear_status_selftest(DevStatusHost* out, cudaStream_t s);

}  // namespace fa
