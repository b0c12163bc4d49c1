// Bandwidth-bound helper kernels of the backward pass (no tensor cores):
//   K2 preprocess: D_i = sum_k dO_ik * O_ik (fp32; O = o + o_lo when the forward's rounding
//                  residual o_lo is given, O read as fp32 when the forward wrote it so),
//                  LSE_i * log2(e), dQ accumulator := 0 (padded rows; not when dQ comes from
//                  the separate pass, which needs no accumulator)
//   K4 dQ convert: dQ = dtype(scale * dQacc)
// Each thread owns one 16-byte vector (8 elements) of a row; the d/8 threads of
// a row sit in one warp and reduce with shuffles. Grid-stride loops keep the
// grid at a few waves of the 152 SMs.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstdint>

#include "ptx.cuh"

namespace fa {

template <bool BF16>
__device__ __forceinline__ void unpack8(const uint4& v, float (&f)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    if constexpr (BF16) {
      __nv_bfloat162 h = *reinterpret_cast<const __nv_bfloat162*>(&w[i]);
      float2 t = __bfloat1622float2(h);
      f[2 * i] = t.x;
      f[2 * i + 1] = t.y;
    } else {
      __half2 h = *reinterpret_cast<const __half2*>(&w[i]);
      float2 t = __half22float2(h);
      f[2 * i] = t.x;
      f[2 * i + 1] = t.y;
    }
  }
}

template <bool BF16>
__device__ __forceinline__ uint32_t pack2f(float lo, float hi) {
  if constexpr (BF16) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
  } else {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
  }
}

// Workspace rows are padded per head: row (bh, r) of D, LSE*log2e and the dQ accumulator sits at
// bh * Npad + r with Npad = N rounded up to 128, so every query step (64 rows) or query tile (128
// rows) of the backward starts 256-byte aligned (a bulk copy needs 16) and stays inside its own head. Padding rows hold D = 0 and
// LSE*log2e = 0 (finite: a masked query still multiplies them by zero).
// VPR = vectors (of 8 elements) per row = d / 8, a power of two <= 32.
template <int VPR, bool BF16>
__global__ void __launch_bounds__(256) fa_bwd_preprocess_kernel(const uint4* __restrict__ o,
                                                                 const uint4* __restrict__ o_lo,
                                                                 const float4* __restrict__ o32,
                                                                 const uint4* __restrict__ dO,
                                                                 const float* __restrict__ lse, float* __restrict__ D,
                                                                 float* __restrict__ lse2, float4* __restrict__ dqacc,
                                                                 int N, int Npad, size_t n_vec_pad) {
  const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
  for (size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n_vec_pad; i += stride) {
    const uint32_t row_pad = static_cast<uint32_t>(i / VPR);
    const uint32_t bh = row_pad / static_cast<uint32_t>(Npad), r = row_pad - bh * static_cast<uint32_t>(Npad);
    const bool real = r < static_cast<uint32_t>(N);
    const size_t row = static_cast<size_t>(bh) * N + r;  // the row in the caller's [B*H*N] layout
    float acc = 0.f;
    if (real) {
      const size_t src = row * VPR + (i % VPR);
      float a[8], b[8];
      if (o32) {  // O given in fp32
        const float4 x = __ldg(&o32[2 * src]), y = __ldg(&o32[2 * src + 1]);
        a[0] = x.x; a[1] = x.y; a[2] = x.z; a[3] = x.w;
        a[4] = y.x; a[5] = y.y; a[6] = y.z; a[7] = y.w;
      } else {
        unpack8<BF16>(__ldg(&o[src]), a);
      }
      unpack8<BF16>(__ldg(&dO[src]), b);
      if (o_lo) {  // O reconstructed to fp32 accuracy: o + residual
        float rr[8];
        unpack8<BF16>(__ldg(&o_lo[src]), rr);
#pragma unroll
        for (int k = 0; k < 8; ++k) a[k] += rr[k];
      }
#pragma unroll
      for (int k = 0; k < 8; ++k) acc = fmaf(a[k], b[k], acc);
    }
    // every lane of a row's VPR-lane group takes the same branch (rows never straddle a group)
#pragma unroll
    for (int off = VPR / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off, VPR);
    if (dqacc) {
      const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
      dqacc[2 * i] = z;
      dqacc[2 * i + 1] = z;
    }
    if ((i % VPR) == 0) {
      D[row_pad] = acc;
      lse2[row_pad] = real ? lse[row] * 1.4426950408889634f : 0.f;
    }
  }
}

// dQ = dtype(scale * accumulator), from the padded accumulator rows to the caller's rows.
template <int VPR, bool BF16>
__global__ void __launch_bounds__(256) fa_bwd_dq_convert_kernel(const float4* __restrict__ dqacc,
                                                                uint4* __restrict__ dq, float scale, int N, int Npad,
                                                                size_t n_vec) {
  const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
  for (size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n_vec; i += stride) {
    const uint32_t row = static_cast<uint32_t>(i / VPR);
    const uint32_t bh = row / static_cast<uint32_t>(N), r = row - bh * static_cast<uint32_t>(N);
    const size_t src = (static_cast<size_t>(bh) * Npad + r) * VPR + (i % VPR);
    const float4 x = dqacc[2 * src], y = dqacc[2 * src + 1];
    uint4 v;
    v.x = pack2f<BF16>(x.x * scale, x.y * scale);
    v.y = pack2f<BF16>(x.z * scale, x.w * scale);
    v.z = pack2f<BF16>(y.x * scale, y.y * scale);
    v.w = pack2f<BF16>(y.z * scale, y.w * scale);
    dq[i] = v;
  }
}

}  // namespace fa
