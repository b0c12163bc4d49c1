// Attention backward main kernel (K3) for sm_103a.
//
// Method (page "transformer模型详解（十）：FlashAttention优化技术", section
// "Re-computation 而非缓存"): nothing of the forward's N x N matrix is kept;
// the backward walks K/V column blocks in an outer loop and Q row blocks in an
// inner loop and recomputes the scores q_i k_j^T / sqrt(d) and the
// probabilities. The probabilities are rebuilt exactly as
// P = exp(scale * S - LSE) from the forward's saved log-sum-exp (the page's
// block-local "softmax(s_ij)" read that way). The gradient steps are
//   dV_j += P^T dO_i;  dP = dO_i V_j^T;  dS = P * (dP - D_i);
//   dK_j += scale * dS^T Q_i;  dQ_i += scale * dS K_j.
//
// This header holds what the backward kernels share: their parameter block,
// the 16-bit packing, the where-codes of their bounded waits and the TMA
// epilogue helper. The kernels: fa_bwd_pipe_kernel (d = 64 and 128,
// fa_bwd_pipe.cuh) and fa_bwd_d256_kernel (d = 256, fa_bwd_d256.cuh).
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "common.cuh"

namespace fa {

struct BwdParams {
  CUtensorMap tm_q, tm_k, tm_v, tm_do, tm_dk, tm_dv;
  const float* lse2;  // [B*H*Npad] LSE * log2(e); row (bh, r) at bh * Npad + r (Npad = N rounded up to 128)
  const float* Dvec;  // [B*H*Npad] rowsum(dO * O), same rows
  float* dqacc;       // [B*H*Npad, d] fp32, same rows (the accumulating dQ path)
  void* dq;           // [B*H*N, d] dtype output, written directly by the separate dQ pass
  void* dk;           // [B*Hkv*N, d] dtype outputs, written directly by kernels that store from registers
  void* dv;
  const int* kv_len;  // optional [B]: keys j >= kv_len[b] are masked for batch b (key padding)
  int N;
  int Npad;           // N rounded up to 128: the per-head row stride of lse2, Dvec and dqacc
  int H, Hkv;         // query heads and K/V heads (Hkv divides H; H / Hkv query heads share one K/V head)
  float scale;
  float scale_log2;
  unsigned long long timeout_ns;
};

// Keys of batch b that exist: min(N, kv_len[b]) (clamped at 0), or N without a key-padding mask.
__device__ __forceinline__ int bwd_key_count(const BwdParams& p, int b) {
  if (!p.kv_len) return p.N;
  const int l = __ldg(p.kv_len + b);
  return l < 0 ? 0 : (l > p.N ? p.N : l);
}

// A key block of K/V head x (of the B*Hkv) feeds G = H / Hkv query heads; its query steps run
// head by head: step `it` is 64-query step it0 + it % n_ith of query head qh0 + it / n_ith.
// GRP = false is plain multi-head attention without a key-padding mask (G = 1, every key exists),
// with all of that known at compile time.
template <bool GRP>
struct BwdGroup {
  int qh0;   // first query head (of the B*H) of the group
  int G;     // query heads per K/V head
  int klen;  // keys that exist for this batch (key padding and N)
  __device__ __forceinline__ BwdGroup(int x, const BwdParams& p) {
    if constexpr (GRP) {
      G = p.H / p.Hkv;
      const int b = x / p.Hkv;
      qh0 = b * p.H + (x - b * p.Hkv) * G;
      klen = bwd_key_count(p, b);
    } else {
      G = 1;
      qh0 = x;
      klen = p.N;
    }
  }
  // query head and 64-query step (within the head) of step `it`
  __device__ __forceinline__ void step(int it, int it0, int n_ith, int& qh, int& qs) const {
    if constexpr (!GRP) {
      qh = qh0;
      qs = it0 + it;
    } else {
      const int gi = G == 1 ? 0 : it / n_ith;
      qh = qh0 + gi;
      qs = it0 + it - gi * n_ith;
    }
  }
};


template <bool BF16>
__device__ __forceinline__ uint32_t bpack2(float lo, float hi) {
  if constexpr (BF16) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
  } else {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
  }
}

// where-codes of the backward's waits and checks (40-59; the forward uses 1-20, decode 31-39)
enum : uint32_t {
  WB_KV = 41, WB_QE = 42, WB_QF = 43, WB_SDP = 44, WB_DS = 45, WB_DQF = 46, WB_DQFREE = 47, WB_DONE = 48, WB_DRAIN = 49,
  WB_ITEM = 50, WB_CLC = 51
};

// Write one 128 x d accumulator (thread = row, TMEM lane) as dtype into a 128-byte-swizzled
// staging tile and store it with TMA at rows [row0, row0 + 128) of head `head`, columns
// [x0, x0 + d); rows past the sequence's end are dropped by the tensor map.
template <int D, bool BF16>
__device__ __forceinline__ void bwd_store_acc(uint32_t tacc, uint8_t* stage, const void* map, int row0, int head, int r,
                                              float mul, uint32_t bar_id, bool ok, volatile uint32_t* abort_flag,
                                              int x0 = 0) {
  if (ok) {
#pragma unroll 1
    for (int c = 0; c < D / 32; ++c) {
      uint32_t u[32];
      tmem_ld32(tacc + 32 * c, u);
#pragma unroll
      for (int g = 0; g < 4; ++g) {
        const int col = 32 * c + 8 * g;
        uint4 v;
        v.x = bpack2<BF16>(__uint_as_float(u[8 * g + 0]) * mul, __uint_as_float(u[8 * g + 1]) * mul);
        v.y = bpack2<BF16>(__uint_as_float(u[8 * g + 2]) * mul, __uint_as_float(u[8 * g + 3]) * mul);
        v.z = bpack2<BF16>(__uint_as_float(u[8 * g + 4]) * mul, __uint_as_float(u[8 * g + 5]) * mul);
        v.w = bpack2<BF16>(__uint_as_float(u[8 * g + 6]) * mul, __uint_as_float(u[8 * g + 7]) * mul);
        const int chunk = col >> 6, unit = (col & 63) >> 3;
        *reinterpret_cast<uint4*>(stage + chunk * (128 * 128) + r * 128 + ((unit ^ (r & 7)) << 4)) = v;
      }
    }
    fence_proxy_async_smem();
  }
  named_bar_sync(bar_id, 128);
  if (r == 0 && ok && *abort_flag == 0u) {
#pragma unroll
    for (int c = 0; c < D / 64; ++c) tma_store_3d(map, smem_u32(stage) + c * (128 * 128), x0 + c * 64, row0, head);
    bulk_commit();
    bulk_wait_read0();
  }
}

}  // namespace fa
