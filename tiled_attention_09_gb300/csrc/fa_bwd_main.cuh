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
// GB300 design. One CTA per (b, h, key tile j of 128 keys); K_j and V_j stay
// in shared memory, dK_j and dV_j accumulate in tensor memory for the whole
// inner loop. Query tiles of BQ rows (64 for d = 128, 128 for d = 64) stream
// through a two-stage TMA ring together with their LSE*log2e and D values.
// Keys are the MMA's M dimension, so S and dP are produced transposed
// (S^T = K_j Q_i^T, dP^T = V_j dO_i^T) with one key per TMEM lane; P^T and
// dS^T then feed dV and dK straight from TMEM. dS^T also goes to shared
// memory (128-byte swizzle) as the operand of the dQ product, whose partial
// tile is added into an fp32 dQ accumulator in global memory with one bulk
// reduce-add per step.
// Roles: warps 0-3 elementwise (P^T, dS^T), warps 4-7 dQ read-out and the dK
// epilogue, warp 8 TMA producer, warp 9 MMA issuer.
// TMEM columns: S^T/P^T at 0, dP^T/dS^T at BQ, dV at 2BQ, dK at 2BQ+d, and two
// 64-column dQ buffers at 2BQ+2d (512 columns in total for d = 64 and 128).
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "common.cuh"

namespace fa {

struct BwdParams {
  CUtensorMap tm_q, tm_k, tm_v, tm_do, tm_dk, tm_dv;
  const float* lse2;  // [B*H*N] LSE * log2(e)
  const float* Dvec;  // [B*H*N] rowsum(dO * O)
  float* dqacc;       // [B*H*N, d] fp32
  void* dk;           // [B*H*N, d] dtype outputs, written directly by kernels that store from registers
  void* dv;
  int N;
  float scale;
  float scale_log2;
  unsigned long long timeout_ns;
};

template <int D>
struct BwdCfg {
  static constexpr int BK = 128;
  static constexpr int BQ = (D == 64) ? 128 : 64;
  static constexpr bool DQ_T = (D != 64);  // dQ^T = K^T dS^T (M = d) when true, dQ = dS K (M = BQ) otherwise
  static constexpr int NCH = D / 64;
  static constexpr int KV_CHUNK = BK * 128;  // 128 rows x 128 bytes
  static constexpr int KV_TILE = BK * D * 2;
  static constexpr int Q_CHUNK = BQ * 128;
  static constexpr int Q_TILE = BQ * D * 2;
  static constexpr int DS_BYTES = BK * BQ * 2;
  static constexpr int DQ_STAGE = BQ * D * 4;
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = OFF_K + KV_TILE;
  static constexpr int OFF_Q = OFF_V + KV_TILE;      // 2 stages
  static constexpr int OFF_DO = OFF_Q + 2 * Q_TILE;  // 2 stages
  static constexpr int OFF_DS = OFF_DO + 2 * Q_TILE;
  static constexpr int OFF_DQ = OFF_DS + DS_BYTES;   // 2 staging buffers
  static constexpr int OFF_LSE = OFF_DQ + 2 * DQ_STAGE;
  static constexpr int OFF_DD = OFF_LSE + 2 * BQ * 4;
  static constexpr int OFF_BAR = OFF_DD + 2 * BQ * 4;
  static constexpr int NBAR = 13;
  static constexpr int SMEM_BYTES = 1024 + OFF_BAR + NBAR * 8 + 16;
  static constexpr int THREADS = 320;
  static constexpr uint32_t S_COL = 0, DP_COL = BQ, DV_COL = 2 * BQ, DK_COL = 2 * BQ + D, DQ_COL = 2 * BQ + 2 * D;
  static_assert(DQ_COL + 128 <= 512, "TMEM budget");
  static_assert(2 * Q_TILE >= KV_TILE, "epilogue staging reuses the Q and dO stages");
  static_assert(SMEM_BYTES <= 227 * 1024, "smem budget");
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

enum : uint32_t {
  WB_KV = 11, WB_QE = 12, WB_QF = 13, WB_SDP = 14, WB_DS = 15, WB_DQF = 16, WB_DQFREE = 17, WB_DONE = 18, WB_DRAIN = 19,
  WB_ITEM = 20, WB_CLC = 21
};

// Write one 128 x d accumulator (thread = row, TMEM lane) as dtype into a 128-byte-swizzled
// staging tile and store it with TMA at rows [row0, row0 + 128), columns [x0, x0 + d).
template <int D, bool BF16>
__device__ __forceinline__ void bwd_store_acc(uint32_t tacc, uint8_t* stage, const void* map, int row0, int r,
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
    for (int c = 0; c < D / 64; ++c) tma_store_2d(map, smem_u32(stage) + c * (128 * 128), x0 + c * 64, row0);
    bulk_commit();
    bulk_wait_read0();
  }
}

template <int D, bool BF16, bool CAUSAL>
__global__ void __launch_bounds__(320, 1) fa_bwd_main_kernel(const __grid_constant__ BwdParams p) {
  using C = BwdCfg<D>;
  constexpr int BQ = C::BQ;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t s0 = smem_u32(smem);
  const uint32_t sK = s0 + C::OFF_K, sV = s0 + C::OFF_V, sQ = s0 + C::OFF_Q, sDO = s0 + C::OFF_DO;
  const uint32_t sDS = s0 + C::OFF_DS, sDQ = s0 + C::OFF_DQ;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  const uint32_t b_kv = smem_u32(&bars[0]);
  auto b_qfull = [&](int s) { return smem_u32(&bars[1 + s]); };
  auto b_qempty = [&](int s) { return smem_u32(&bars[3 + s]); };
  const uint32_t b_sdp = smem_u32(&bars[5]);
  const uint32_t b_ds = smem_u32(&bars[6]);
  auto b_dqfull = [&](int b) { return smem_u32(&bars[7 + b]); };
  auto b_dqfree = [&](int b) { return smem_u32(&bars[9 + b]); };
  const uint32_t b_done = smem_u32(&bars[11]);
  const uint32_t b_drain = smem_u32(&bars[12]);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(&bars[C::NBAR]);
  volatile uint32_t* abort_flag = tmem_slot + 1;

  const int warp = threadIdx.x >> 5;
  const int N = p.N;
  const int bh = blockIdx.x;
  const int key0 = blockIdx.y * 128;
  const int row_base = bh * N;
  const int it0 = CAUSAL ? (key0 / BQ) : 0;
  const int n_it = N / BQ - it0;

  if (threadIdx.x == 0) {
    mbar_init(b_kv, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(b_qfull(s), 1);
      mbar_init(b_qempty(s), 1);
      mbar_init(b_dqfull(s), 1);
      mbar_init(b_dqfree(s), 128);
    }
    mbar_init(b_sdp, 1);
    mbar_init(b_ds, 128);
    mbar_init(b_done, 1);
    mbar_init(b_drain, 1);
    *abort_flag = 0u;
    mbar_fence_init();
    fence_proxy_async_smem();
  }
  if (warp == 9) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 8) {
    // ------------------------------------------------------------ producer
    if (elect_one()) {
      tma_prefetch_desc(&p.tm_q);
      tma_prefetch_desc(&p.tm_do);
      mbar_arrive_expect_tx(b_kv, 2 * C::KV_TILE);
#pragma unroll
      for (int c = 0; c < C::NCH; ++c) {
        tma_load_2d(sK + c * C::KV_CHUNK, &p.tm_k, b_kv, c * 64, row_base + key0);
        tma_load_2d(sV + c * C::KV_CHUNK, &p.tm_v, b_kv, c * 64, row_base + key0);
      }
      int issued = 0;
      for (int it = 0; it < n_it; ++it) {
        const int s = it & 1, use = it >> 1;
        if (use > 0 && !wait_bar(b_qempty(s), (use - 1) & 1, p.timeout_ns, abort_flag, WB_QE)) break;
        const int qrow = row_base + (it0 + it) * BQ;
        mbar_arrive_expect_tx(b_qfull(s), 2 * C::Q_TILE + 2 * BQ * 4);
#pragma unroll
        for (int c = 0; c < C::NCH; ++c) {
          tma_load_2d(sQ + s * C::Q_TILE + c * C::Q_CHUNK, &p.tm_q, b_qfull(s), c * 64, qrow);
          tma_load_2d(sDO + s * C::Q_TILE + c * C::Q_CHUNK, &p.tm_do, b_qfull(s), c * 64, qrow);
        }
        bulk_load(s0 + C::OFF_LSE + s * BQ * 4, p.lse2 + qrow, BQ * 4, b_qfull(s));
        bulk_load(s0 + C::OFF_DD + s * BQ * 4, p.Dvec + qrow, BQ * 4, b_qfull(s));
        ++issued;
      }
      wait_bar(b_kv, 0, p.timeout_ns, abort_flag, WB_DRAIN);
      for (int it = (issued > 2 ? issued - 2 : 0); it < issued; ++it)
        wait_bar(b_qfull(it & 1), (it >> 1) & 1, p.timeout_ns, abort_flag, WB_DRAIN);
    }
    __syncwarp();
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    if (elect_one()) {
      constexpr uint32_t idesc_sdp = make_idesc(128, BQ, BF16, false, false);
      constexpr uint32_t idesc_acc = make_idesc(128, D, BF16, false, true);
      constexpr uint32_t idesc_dq = C::DQ_T ? make_idesc(128, BQ, BF16, true, true) : make_idesc(128, D, BF16, true, true);
      bool ok = wait_bar(b_kv, 0, p.timeout_ns, abort_flag, WB_KV);
      for (int it = 0; ok && it < n_it; ++it) {
        const int s = it & 1, use = it >> 1;
        if (!wait_bar(b_qfull(s), use & 1, p.timeout_ns, abort_flag, WB_QF)) break;
        tc_fence_after();
        const uint32_t sQs = sQ + s * C::Q_TILE, sDOs = sDO + s * C::Q_TILE;
        // S^T = K_j Q_i^T and dP^T = V_j dO_i^T  (M = 128 keys, N = BQ, K = d)
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t oa = (kk >> 2) * C::KV_CHUNK + (kk & 3) * 32;
          const uint32_t ob = (kk >> 2) * C::Q_CHUNK + (kk & 3) * 32;
          mma_ss(tmem + C::S_COL, make_sdesc(sK + oa, 16, 1024), make_sdesc(sQs + ob, 16, 1024), idesc_sdp,
                 kk > 0 ? 1u : 0u);
        }
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t oa = (kk >> 2) * C::KV_CHUNK + (kk & 3) * 32;
          const uint32_t ob = (kk >> 2) * C::Q_CHUNK + (kk & 3) * 32;
          mma_ss(tmem + C::DP_COL, make_sdesc(sV + oa, 16, 1024), make_sdesc(sDOs + ob, 16, 1024), idesc_sdp,
                 kk > 0 ? 1u : 0u);
        }
        mma_commit(b_sdp);
        if (!wait_bar(b_ds, it & 1, p.timeout_ns, abort_flag, WB_DS)) break;
        tc_fence_after();
        // dV += P^T dO_i ; dK += dS^T Q_i   (M = 128 keys, N = d, K = BQ; A from TMEM, B MN-major)
#pragma unroll
        for (int kk = 0; kk < BQ / 16; ++kk)
          mma_ts(tmem + C::DV_COL, tmem + C::S_COL + kk * 8, make_sdesc(sDOs + kk * 2048, C::Q_CHUNK, 1024),
                 idesc_acc, (it > 0 || kk > 0) ? 1u : 0u);
#pragma unroll
        for (int kk = 0; kk < BQ / 16; ++kk)
          mma_ts(tmem + C::DK_COL, tmem + C::DP_COL + kk * 8, make_sdesc(sQs + kk * 2048, C::Q_CHUNK, 1024),
                 idesc_acc, (it > 0 || kk > 0) ? 1u : 0u);
        mma_commit(b_qempty(s));
        // dQ partial into TMEM buffer it&1 (K = 128 keys, both operands MN-major)
        const int b = it & 1, ub = it >> 1;
        if (ub > 0 && !wait_bar(b_dqfree(b), (ub - 1) & 1, p.timeout_ns, abort_flag, WB_DQFREE)) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          uint64_t da, db;
          if constexpr (C::DQ_T) {  // dQ^T[d][q] = sum_k K[k][d] dS^T[k][q]
            da = make_sdesc(sK + kk * 2048, C::KV_CHUNK, 1024);
            db = make_sdesc(sDS + kk * 2048, 128 * 128, 1024);
          } else {  // dQ[q][d] = sum_k dS^T[k][q] K[k][d]
            da = make_sdesc(sDS + kk * 2048, 128 * 128, 1024);
            db = make_sdesc(sK + kk * 2048, C::KV_CHUNK, 1024);
          }
          mma_ss(tmem + C::DQ_COL + 64 * b, da, db, idesc_dq, kk > 0 ? 1u : 0u);
        }
        mma_commit(b_dqfull(b));
      }
      mma_commit(b_done);
      mma_commit(b_drain);
      wait_bar(b_drain, 0, p.timeout_ns, abort_flag, WB_DRAIN);
    }
    __syncwarp();
  } else if (warp < 4) {
    // ------------------------------------------------------------ elementwise: P^T, dS^T
    const int k = threadIdx.x;  // key within the tile == TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
    const uint32_t tS = tmem + lane_off + C::S_COL, tDP = tmem + lane_off + C::DP_COL;
    const float sl2 = p.scale_log2;
    bool ok = true;
    for (int it = 0; it < n_it; ++it) {
      const int s = it & 1;
      if (!__all_sync(0xffffffffu, wait_bar(b_sdp, it & 1, p.timeout_ns, abort_flag, WB_SDP))) {
        ok = false;
        break;
      }
      // LSE/D of this stage were landed by the producer on q_full[s]; acquire them here too.
      if (!__all_sync(0xffffffffu, wait_bar(b_qfull(s), (it >> 1) & 1, p.timeout_ns, abort_flag, WB_QF))) {
        ok = false;
        break;
      }
      tc_fence_after();
      const float* lse_s = reinterpret_cast<const float*>(smem + C::OFF_LSE + s * BQ * 4);
      const float* dd_s = reinterpret_cast<const float*>(smem + C::OFF_DD + s * BQ * 4);
      const int q0 = (it0 + it) * BQ;  // first query of the tile
      const bool need_mask = CAUSAL && (q0 < key0 + 127);
      const int kq = key0 + k - q0;  // masked where column c < kq (key > query)
#pragma unroll
      for (int h = 0; h < BQ / 64; ++h) {
        float pv[64];
        {
          uint32_t u0[32], u1[32];
          tmem_ld32(tS + 64 * h, u0);
          tmem_ld32(tS + 64 * h + 32, u1);
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            pv[c] = ex2_approx(fmaf(__uint_as_float(u0[c]), sl2, -lse_s[64 * h + c]));
            pv[32 + c] = ex2_approx(fmaf(__uint_as_float(u1[c]), sl2, -lse_s[64 * h + 32 + c]));
          }
        }
        if (need_mask) {
#pragma unroll
          for (int c = 0; c < 64; ++c) pv[c] = (64 * h + c < kq) ? 0.f : pv[c];
        }
        {
          uint32_t pk[32];
#pragma unroll
          for (int c = 0; c < 32; ++c) pk[c] = bpack2<BF16>(pv[2 * c], pv[2 * c + 1]);
          tmem_st32(tS + 32 * h, pk);
        }
        uint32_t dk32[32];
        {
          uint32_t u0[32], u1[32];
          tmem_ld32(tDP + 64 * h, u0);
          tmem_ld32(tDP + 64 * h + 32, u1);
#pragma unroll
          for (int c = 0; c < 16; ++c) {
            const float a0 = pv[2 * c] * (__uint_as_float(u0[2 * c]) - dd_s[64 * h + 2 * c]);
            const float a1 = pv[2 * c + 1] * (__uint_as_float(u0[2 * c + 1]) - dd_s[64 * h + 2 * c + 1]);
            dk32[c] = bpack2<BF16>(a0, a1);
            const float b0 = pv[32 + 2 * c] * (__uint_as_float(u1[2 * c]) - dd_s[64 * h + 32 + 2 * c]);
            const float b1 = pv[33 + 2 * c] * (__uint_as_float(u1[2 * c + 1]) - dd_s[64 * h + 33 + 2 * c]);
            dk32[16 + c] = bpack2<BF16>(b0, b1);
          }
        }
        tmem_st32(tDP + 32 * h, dk32);
        // dS^T row k, queries 64h .. 64h+63: one 128-byte swizzled row of chunk h
        uint8_t* row = smem + C::OFF_DS + h * (128 * 128) + k * 128;
#pragma unroll
        for (int u = 0; u < 8; ++u)
          *reinterpret_cast<uint4*>(row + ((u ^ (k & 7)) << 4)) =
              make_uint4(dk32[4 * u], dk32[4 * u + 1], dk32[4 * u + 2], dk32[4 * u + 3]);
      }
      fence_proxy_async_smem();
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(b_ds);
    }
    if (ok) ok = __all_sync(0xffffffffu, wait_bar(b_done, 0, p.timeout_ns, abort_flag, WB_DONE));
    if (ok) tc_fence_after();
    bwd_store_acc<D, BF16>(tmem + lane_off + C::DV_COL, smem + C::OFF_Q, &p.tm_dv, row_base + key0, k, 1.0f, 1, ok,
                           abort_flag);
  } else {
    // ------------------------------------------------------------ dQ read-out, then dK epilogue
    const int t = threadIdx.x - 128;  // TMEM lane: d index (dQ^T) or query index (dQ)
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    bool ok = true;
    // Every warp runs all n_it steps and both named barriers of each step, even after an
    // abort (waits then return at once), so no warp of this group can be left at a barrier.
    for (int it = 0; it < n_it; ++it) {
      const int b = it & 1;
      ok = ok && __all_sync(0xffffffffu, wait_bar(b_dqfull(b), (it >> 1) & 1, p.timeout_ns, abort_flag, WB_DQF));
      uint32_t u0[32], u1[32];
      if (ok) {
        tc_fence_after();
        tmem_ld32(tmem + lane_off + C::DQ_COL + 64 * b, u0);
        tmem_ld32(tmem + lane_off + C::DQ_COL + 64 * b + 32, u1);
        tc_fence_before();
        mbar_arrive(b_dqfree(b));
      } else {
#pragma unroll
        for (int c = 0; c < 32; ++c) u0[c] = u1[c] = 0u;
      }
      // staging buffer b is free once the reduce issued two steps ago has read it
      if (t == 0) asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
      named_bar_sync(2, 128);
      float* st = reinterpret_cast<float*>(smem + C::OFF_DQ + b * C::DQ_STAGE);
      if constexpr (C::DQ_T) {  // lane t = d index; column c = query
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          st[c * D + t] = __uint_as_float(u0[c]);
          st[(32 + c) * D + t] = __uint_as_float(u1[c]);
        }
      } else {  // lane t = query; column c = d index; rotate the 16-byte slots to spread banks
#pragma unroll
        for (int cc = 0; cc < 16; ++cc) {
          const int c4 = (cc + t) & 15;
          float4 v;
          if (c4 < 8) {
            v = make_float4(__uint_as_float(u0[4 * c4]), __uint_as_float(u0[4 * c4 + 1]),
                            __uint_as_float(u0[4 * c4 + 2]), __uint_as_float(u0[4 * c4 + 3]));
          } else {
            const int e = 4 * (c4 - 8);
            v = make_float4(__uint_as_float(u1[e]), __uint_as_float(u1[e + 1]), __uint_as_float(u1[e + 2]),
                            __uint_as_float(u1[e + 3]));
          }
          *reinterpret_cast<float4*>(st + t * 64 + 4 * c4) = v;
        }
      }
      fence_proxy_async_smem();
      named_bar_sync(2, 128);
      if (t == 0 && ok && *abort_flag == 0u) {
        bulk_reduce_add_f32(p.dqacc + static_cast<size_t>(row_base + (it0 + it) * BQ) * D,
                            sDQ + b * C::DQ_STAGE, C::DQ_STAGE);
        bulk_commit();
      }
    }
    if (t == 0) bulk_wait0();
    if (ok) ok = __all_sync(0xffffffffu, wait_bar(b_done, 0, p.timeout_ns, abort_flag, WB_DONE));
    if (ok) tc_fence_after();
    bwd_store_acc<D, BF16>(tmem + lane_off + C::DK_COL, smem + C::OFF_DO, &p.tm_dk, row_base + key0, t, p.scale, 3,
                           ok, abort_flag);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace fa
