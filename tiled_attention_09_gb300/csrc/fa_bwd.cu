// Attention backward for sm_103a: preprocess (K2), main kernel (K3), dQ convert (K4).
#include <cuda.h>

#include "common.cuh"
#include "fa_bwd_aux.cuh"
#include "fa_bwd_main.cuh"
#include "fa_bwd_d256.cuh"
#include "fa_bwd_pipe.cuh"
#include "fa_bwd_dq.cuh"
#include "launch.h"

namespace fa {
namespace {

int grid_for(size_t n_vec) {
  size_t blocks = (n_vec + 255) / 256;
  const size_t cap = 152 * 16;
  return static_cast<int>(blocks < cap ? blocks : cap);
}

template <int VPR>
cudaError_t launch_pre_t(const BwdArgs& a) {
  const size_t n_vec_pad = static_cast<size_t>(a.B) * a.H * a.Npad * VPR;
  float4* dqacc = a.dq_pass ? nullptr : reinterpret_cast<float4*>(a.ws_dqacc);  // the pass needs no accumulator
  if (a.bf16)
    return launch_kernel(fa_bwd_preprocess_kernel<VPR, true>, dim3(grid_for(n_vec_pad)), dim3(256), 0, a.stream,
                         static_cast<const uint4*>(a.o), static_cast<const uint4*>(a.o_lo),
                         a.o_f32 ? static_cast<const float4*>(a.o) : nullptr, static_cast<const uint4*>(a.dO),
                         a.lse, a.ws_D, a.ws_lse2, dqacc, a.N, a.Npad, n_vec_pad);
  return launch_kernel(fa_bwd_preprocess_kernel<VPR, false>, dim3(grid_for(n_vec_pad)), dim3(256), 0, a.stream,
                       static_cast<const uint4*>(a.o), static_cast<const uint4*>(a.o_lo),
                       a.o_f32 ? static_cast<const float4*>(a.o) : nullptr, static_cast<const uint4*>(a.dO),
                       a.lse, a.ws_D, a.ws_lse2, dqacc, a.N, a.Npad, n_vec_pad);
}
template <int VPR>
cudaError_t launch_convert_t(const BwdArgs& a) {
  const size_t n_vec = static_cast<size_t>(a.B) * a.H * a.N * VPR;
  if (a.bf16)
    return launch_kernel(fa_bwd_dq_convert_kernel<VPR, true>, dim3(grid_for(n_vec)), dim3(256), 0, a.stream,
                         reinterpret_cast<const float4*>(a.ws_dqacc), static_cast<uint4*>(a.dq), a.scale, a.N,
                         a.Npad, n_vec);
  return launch_kernel(fa_bwd_dq_convert_kernel<VPR, false>, dim3(grid_for(n_vec)), dim3(256), 0, a.stream,
                       reinterpret_cast<const float4*>(a.ws_dqacc), static_cast<uint4*>(a.dq), a.scale, a.N, a.Npad,
                       n_vec);
}

}  // namespace

cudaError_t launch_bwd_preprocess(const BwdArgs& a) {
  switch (a.d) {
    case 64: return launch_pre_t<8>(a);
    case 128: return launch_pre_t<16>(a);
    case 256: return launch_pre_t<32>(a);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_bwd_dq_convert(const BwdArgs& a) {
  switch (a.d) {
    case 64: return launch_convert_t<8>(a);
    case 128: return launch_convert_t<16>(a);
    case 256: return launch_convert_t<32>(a);
  }
  return cudaErrorInvalidValue;
}

namespace {
BwdParams bwd_params(const BwdArgs& a) {
  BwdParams p;
  p.tm_q = a.tm_q;
  p.tm_k = a.tm_k;
  p.tm_v = a.tm_v;
  p.tm_do = a.tm_do;
  p.tm_dk = a.tm_dk;
  p.tm_dv = a.tm_dv;
  p.lse2 = a.ws_lse2;
  p.Dvec = a.ws_D;
  p.dqacc = a.ws_dqacc;
  p.dq = a.dq;
  p.dk = a.dk;
  p.dv = a.dv;
  p.kv_len = a.kv_len;
  p.N = a.N;
  p.Npad = a.Npad;
  p.H = a.H;
  p.Hkv = a.Hkv;
  p.scale = a.scale;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  p.timeout_ns = a.timeout_ns;
  return p;
}

template <int D, bool BF16, bool CAUSAL, bool GRP>
cudaError_t launch_dq_t(const BwdArgs& a) {
  using C = BwdDqCfg<D>;
  auto kern = fa_bwd_dq_kernel<D, BF16, CAUSAL, GRP>;
  static std::atomic<unsigned long long> attr_done{0};
  cudaError_t e = smem_attr_once(reinterpret_cast<const void*>(kern), C::SMEM_BYTES, attr_done);
  if (e != cudaSuccess) return e;
  const BwdParams p = bwd_params(a);
  dim3 grid(a.B * a.H, (a.N + 127) / 128, 1);  // 128-row query tiles of each query head
  return launch_kernel(kern, grid, dim3(C::THREADS), C::SMEM_BYTES, a.stream, p);
}

template <int D, bool BF16, bool CAUSAL, bool GRP, bool DQACC>
cudaError_t launch_pipe_t(const BwdArgs& a) {
  using C = BwdPipeCfg<D>;
  auto kern = fa_bwd_pipe_kernel<D, BF16, CAUSAL, GRP, DQACC>;
  static std::atomic<unsigned long long> attr_done{0};
  cudaError_t e = smem_attr_once(reinterpret_cast<const void*>(kern), C::SMEM_BYTES, attr_done);
  if (e != cudaSuccess) return e;
  static int checked = 0;  // 1: the compiled register count matches the kernel's register split
  if (!checked) {
    cudaFuncAttributes fa_attr;
    if ((e = cudaFuncGetAttributes(&fa_attr, kern)) != cudaSuccess) return e;
    if (fa_attr.numRegs != C::LAUNCH_REGS) return cudaErrorInvalidConfiguration;
    checked = 1;
  }
  const BwdParams p = bwd_params(a);
  dim3 grid(a.B * a.Hkv, (a.N + 127) / 128, 1);  // key blocks of each K/V head; the last may run past N
  e = launch_kernel(kern, grid, dim3(C::THREADS), C::SMEM_BYTES, a.stream, p);
  if (e != cudaSuccess || a.dq == nullptr) return e;
  return DQACC ? launch_bwd_dq_convert(a) : launch_bwd_dq_pass(a);
}
template <bool BF16, bool CAUSAL>
cudaError_t launch_d256_t(const BwdArgs& a) {
  using C = BwdD256Cfg;
  auto kern = fa_bwd_d256_kernel<BF16, CAUSAL>;
  static std::atomic<unsigned long long> attr_done{0};
  cudaError_t e = smem_attr_once(reinterpret_cast<const void*>(kern), C::SMEM_BYTES, attr_done);
  if (e != cudaSuccess) return e;
  const BwdParams p = bwd_params(a);
  dim3 grid(a.B * a.Hkv, (a.N + 127) / 128, 1);  // key blocks of each K/V head; the last may run past N
  e = launch_kernel(kern, grid, dim3(C::THREADS), C::SMEM_BYTES, a.stream, p);
  if (e != cudaSuccess || a.dq == nullptr) return e;
  return launch_bwd_dq_convert(a);
}
template <int D, bool DQACC>
cudaError_t launch_pipe_dm(const BwdArgs& a) {
  const bool grp = a.Hkv != a.H || a.kv_len != nullptr;  // the general form only where it is needed
  if (a.bf16) {
    if (a.causal)
      return grp ? launch_pipe_t<D, true, true, true, DQACC>(a) : launch_pipe_t<D, true, true, false, DQACC>(a);
    return grp ? launch_pipe_t<D, true, false, true, DQACC>(a) : launch_pipe_t<D, true, false, false, DQACC>(a);
  }
  if (a.causal)
    return grp ? launch_pipe_t<D, false, true, true, DQACC>(a) : launch_pipe_t<D, false, true, false, DQACC>(a);
  return grp ? launch_pipe_t<D, false, false, true, DQACC>(a) : launch_pipe_t<D, false, false, false, DQACC>(a);
}
template <int D>
cudaError_t launch_pipe_d(const BwdArgs& a) {
  return a.dq_pass ? launch_pipe_dm<D, false>(a) : launch_pipe_dm<D, true>(a);
}
template <int D>
cudaError_t launch_dq_d(const BwdArgs& a) {
  const bool grp = a.Hkv != a.H || a.kv_len != nullptr;
  if (a.bf16) {
    if (a.causal) return grp ? launch_dq_t<D, true, true, true>(a) : launch_dq_t<D, true, true, false>(a);
    return grp ? launch_dq_t<D, true, false, true>(a) : launch_dq_t<D, true, false, false>(a);
  }
  if (a.causal) return grp ? launch_dq_t<D, false, true, true>(a) : launch_dq_t<D, false, true, false>(a);
  return grp ? launch_dq_t<D, false, false, true>(a) : launch_dq_t<D, false, false, false>(a);
}
}  // namespace

cudaError_t launch_bwd_dq_pass(const BwdArgs& a) {
  if (a.d == 128) return launch_dq_d<128>(a);
  if (a.d == 64) return launch_dq_d<64>(a);
  return cudaErrorNotSupported;  // d = 256 accumulates dQ in its main kernel
}

cudaError_t launch_bwd_main(const BwdArgs& a) {
  if (a.d == 256) {  // head-dimension split: two passes per key block
    if (a.bf16) return a.causal ? launch_d256_t<true, true>(a) : launch_d256_t<true, false>(a);
    return a.causal ? launch_d256_t<false, true>(a) : launch_d256_t<false, false>(a);
  }
  if (a.d == 128) return launch_pipe_d<128>(a);  // software-pipelined, persistent kernel
  if (a.d == 64) return launch_pipe_d<64>(a);    // the same kernel, K^T zero-padded to 128 rows for dQ^T
  return cudaErrorNotSupported;
}

cudaError_t read_clear_status_bwd(DevStatusHost* out, cudaStream_t s) {
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
