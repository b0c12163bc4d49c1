// Attention backward main kernel, software-pipelined variant for d = 128 (K3).
//
// Same method and per-step arithmetic as fa_bwd_main_kernel (page
// "transformer模型详解（十）：FlashAttention优化技术", section "Re-computation 而非缓存":
// outer loop over K/V column blocks, inner loop over Q row blocks, P rebuilt from
// the saved LSE). What changes is the schedule, so that the tensor core never
// waits for the elementwise warps:
//   * S^T and dP^T of query tile i go to one of two TMEM buffers (i & 1);
//   * S^T(i+1), dP^T(i+1) are issued into the other buffer *before* the
//     issuers wait for P^T(i), dS^T(i), so the tensor core computes the next
//     scores while the elementwise warps turn the current ones into P and dS;
//   * dQ^T(i) = K^T dS^T(i) is written over S^T(i)'s columns once dV(i) has
//     read P^T(i) from them, and read out before S^T(i+2) reuses the buffer;
//   * dS^T goes to a double-buffered shared-memory tile (the dQ operand), and
//     Q, dO, LSE*log2e, D stream through a three-stage TMA ring.
// TMEM (512 columns): buffer b at 128b holds S^T/P^T (cols 0-63, then dQ^T)
// and dP^T/dS^T (cols 64-127); dV at 256, dK at 384. Packed 16-bit P^T of
// queries 32g..32g+31 sits in columns 32g..32g+15 (dS^T likewise from 64).
// Roles (16 warps, 4 per SM sub-partition): warps 0-7 elementwise, in two
// groups that each own 32 of the tile's 64 query columns; warps 8-11 dQ
// read-out and the dK epilogue; warp 12 TMA producer; warps 13-15 MMA issuers
// (S^T + dV, dP^T + dK, dQ^T), since one thread cannot issue fast enough.
#pragma once
#include "fa_bwd_main.cuh"

namespace fa {

struct BwdPipeCfg {
  static constexpr int D = 128, BK = 128, BQ = 64, NCH = 2, NSTAGE = 3;
  static constexpr int KV_CHUNK = BK * 128;  // 16 KB: 128 rows x 128 bytes
  static constexpr int KV_TILE = BK * D * 2;  // 32 KB
  static constexpr int Q_CHUNK = BQ * 128;    // 8 KB
  static constexpr int Q_TILE = BQ * D * 2;   // 16 KB
  static constexpr int DS_TILE = BK * BQ * 2;  // 16 KB: dS^T [128 keys][64 queries]
  static constexpr int DQ_STAGE = BQ * D * 4;  // 32 KB fp32 [64 queries][128]
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = OFF_K + KV_TILE;
  static constexpr int OFF_Q = OFF_V + KV_TILE;             // NSTAGE stages
  static constexpr int OFF_DO = OFF_Q + NSTAGE * Q_TILE;    // NSTAGE stages
  static constexpr int OFF_DS = OFF_DO + NSTAGE * Q_TILE;   // 2 buffers
  static constexpr int OFF_DQ = OFF_DS + 2 * DS_TILE;       // 1 staging buffer
  static constexpr int OFF_LSE = OFF_DQ + DQ_STAGE;         // NSTAGE x BQ floats
  static constexpr int OFF_DD = OFF_LSE + NSTAGE * BQ * 4;  // NSTAGE x BQ floats
  static constexpr int OFF_BAR = OFF_DD + NSTAGE * BQ * 4;
  // bars: kv, q_full[3], q_empty[3], sdp_full[2], ds_full[2], dq_full[2], dq_free[2], dv_done[2], done,
  // drain[3]
  static constexpr int NBAR = 1 + 2 * NSTAGE + 10 + 1 + 3;
  static constexpr int SMEM_BYTES = 1024 + OFF_BAR + NBAR * 8 + 16;
  static constexpr int THREADS = 512;
  __host__ __device__ static constexpr uint32_t BUF(int b) { return 128u * b; }
  static constexpr uint32_t DV_COL = 256, DK_COL = 384;
  static_assert(NSTAGE * Q_TILE >= KV_TILE, "epilogue staging reuses the Q and dO stages");
  static_assert(SMEM_BYTES <= 232448, "smem budget");
};

template <bool BF16, bool CAUSAL>
__global__ void __launch_bounds__(512, 1) fa_bwd_pipe_kernel(const __grid_constant__ BwdParams p) {
  using C = BwdPipeCfg;
  constexpr int BQ = C::BQ, D = C::D, NS = C::NSTAGE;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t s0 = smem_u32(smem);
  const uint32_t sK = s0 + C::OFF_K, sV = s0 + C::OFF_V, sQ = s0 + C::OFF_Q, sDO = s0 + C::OFF_DO;
  const uint32_t sDS = s0 + C::OFF_DS, sDQ = s0 + C::OFF_DQ;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  const uint32_t b_kv = smem_u32(&bars[0]);
  auto b_qfull = [&](int s) { return smem_u32(&bars[1 + s]); };
  auto b_qempty = [&](int s) { return smem_u32(&bars[1 + NS + s]); };
  auto b_sdp = [&](int b) { return smem_u32(&bars[1 + 2 * NS + b]); };
  auto b_ds = [&](int b) { return smem_u32(&bars[3 + 2 * NS + b]); };
  auto b_dqfull = [&](int b) { return smem_u32(&bars[5 + 2 * NS + b]); };
  auto b_dqfree = [&](int b) { return smem_u32(&bars[7 + 2 * NS + b]); };
  auto b_dvdone = [&](int b) { return smem_u32(&bars[9 + 2 * NS + b]); };
  const uint32_t b_done = smem_u32(&bars[11 + 2 * NS]);
  auto b_drain = [&](int i) { return smem_u32(&bars[12 + 2 * NS + i]); };
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
    for (int s = 0; s < NS; ++s) {
      mbar_init(b_qfull(s), 1);
      mbar_init(b_qempty(s), 2);  // released by issuers A (after dV) and B (after dK)
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(b_sdp(b), 2);  // S^T from issuer A, dP^T from issuer B
      mbar_init(b_ds(b), 256);
      mbar_init(b_dqfull(b), 1);
      mbar_init(b_dqfree(b), 128);
      mbar_init(b_dvdone(b), 1);
    }
    mbar_init(b_done, 3);
    for (int i = 0; i < 3; ++i) mbar_init(b_drain(i), 1);
    *abort_flag = 0u;
    mbar_fence_init();
    fence_proxy_async_smem();
  }
  if (warp == 13) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 12) {
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
        const int s = it % NS, use = it / NS;
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
      for (int it = (issued > NS ? issued - NS : 0); it < issued; ++it)
        wait_bar(b_qfull(it % NS), (it / NS) & 1, p.timeout_ns, abort_flag, WB_DRAIN);
    }
    __syncwarp();
  } else if (warp >= 13) {
    // ------------------------------------------------------------ MMA issuers
    // One thread issues a tcgen05.mma only every ~100+ cycles, so the step's 32 MMAs are spread
    // over three warps: A = S^T and dV, B = dP^T and dK, C = dQ^T. A's and B's accumulators are
    // disjoint; C writes dQ^T over the S^T/P^T columns of the step, so it first waits for dV
    // (issuer A) to have read P^T there (dv_done). A only re-fills a buffer after warps 8-11 have
    // read the dQ^T that C left in it (dq_free).
    const int role = warp - 13;
    if (elect_one()) {
      constexpr uint32_t idesc_sdp = make_idesc(128, BQ, BF16, false, false);
      constexpr uint32_t idesc_acc = make_idesc(128, D, BF16, false, true);
      constexpr uint32_t idesc_dq = make_idesc(128, BQ, BF16, true, true);
      // Descriptors are built once; a K or row step only adds a constant to the 14-bit start-address
      // field (start >> 4), which never carries out of it (shared memory is below 256 KB).
      const uint64_t dKV_k = make_sdesc(role == 0 ? sK : sV, 16, 1024);            // A: K, B: V (K-major)
      const uint64_t dQO_k = make_sdesc(role == 0 ? sQ : sDO, 16, 1024);           // A: Q, B: dO (K-major)
      const uint64_t dOQ_mn = make_sdesc(role == 0 ? sDO : sQ, C::Q_CHUNK, 1024);  // A: dO, B: Q (MN-major)
      const uint64_t dK_mn = make_sdesc(sK, C::KV_CHUNK, 1024);                    // C: K^T (MN-major)
      const uint64_t dDS_mn = make_sdesc(sDS, 128 * 128, 1024);                    // C: dS^T (MN-major)
      const uint32_t col = role == 0 ? 0u : 64u;  // A: S^T / P^T half of a buffer, B: dP^T / dS^T half
      const uint32_t acc_col = role == 0 ? C::DV_COL : C::DK_COL;
      // A: S^T(i) = K_j Q_i^T ; B: dP^T(i) = V_j dO_i^T  (M = 128 keys, N = 64, K = d) into buffer i & 1
      auto issue_score = [&](int it) {
        const uint64_t so = static_cast<uint64_t>((it % NS) * C::Q_TILE) >> 4;
        const uint32_t tb = tmem + C::BUF(it & 1) + col;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint64_t oa = ((kk >> 2) * C::KV_CHUNK + (kk & 3) * 32) >> 4;
          const uint64_t ob = ((kk >> 2) * C::Q_CHUNK + (kk & 3) * 32) >> 4;
          mma_ss(tb, dKV_k + oa, dQO_k + so + ob, idesc_sdp, kk > 0 ? 1u : 0u);
        }
        mma_commit(b_sdp(it & 1));
      };
      bool ok = true;
      if (role < 2) {
        ok = wait_bar(b_kv, 0, p.timeout_ns, abort_flag, WB_KV) &&
             wait_bar(b_qfull(0), 0, p.timeout_ns, abort_flag, WB_QF);
        if (ok) {
          tc_fence_after();
          issue_score(0);
        }
        for (int it = 0; ok && it < n_it; ++it) {
          const int b = it & 1;
          if (it + 1 < n_it) {
            const int nx = it + 1, u1 = nx >> 1;
            if (!wait_bar(b_qfull(nx % NS), (nx / NS) & 1, p.timeout_ns, abort_flag, WB_QF)) break;
            // A: buffer nx & 1 still holds dQ^T(it - 1) until warps 8-11 have read it out
            if (role == 0 && u1 >= 1 &&
                !wait_bar(b_dqfree(nx & 1), (u1 - 1) & 1, p.timeout_ns, abort_flag, WB_DQFREE))
              break;
            tc_fence_after();
            issue_score(nx);
          }
          if (!wait_bar(b_ds(b), (it >> 1) & 1, p.timeout_ns, abort_flag, WB_DS)) break;
          tc_fence_after();
          const int s = it % NS;
          const uint64_t so = static_cast<uint64_t>(s * C::Q_TILE) >> 4;
          const uint32_t tb = tmem + C::BUF(b) + col;
          const uint32_t acc0 = it > 0 ? 1u : 0u;
          // A: dV += P^T dO_i ; B: dK += dS^T Q_i  (M = 128 keys, N = d, K = 64; A from TMEM, B MN-major).
          // Packed P^T / dS^T of queries 16kk .. 16kk+15 sit at column (kk / 2) * 32 + (kk % 2) * 8.
#pragma unroll
          for (int kk = 0; kk < BQ / 16; ++kk)
            mma_ts(tmem + acc_col, tb + (kk >> 1) * 32 + (kk & 1) * 8, dOQ_mn + so + ((kk * 2048) >> 4), idesc_acc,
                   kk > 0 ? 1u : acc0);
          mma_commit(b_qempty(s));
          if (role == 0) mma_commit(b_dvdone(b));
        }
      } else {
        // C: dQ^T(i) = K_j^T dS^T(i) over S^T(i)'s columns (M = d, N = 64 queries, K = 128 keys)
        for (int it = 0; ok && it < n_it; ++it) {
          const int b = it & 1;
          if (!wait_bar(b_ds(b), (it >> 1) & 1, p.timeout_ns, abort_flag, WB_DS)) break;
          if (!wait_bar(b_dvdone(b), (it >> 1) & 1, p.timeout_ns, abort_flag, WB_DS)) break;
          tc_fence_after();
          const uint32_t tb = tmem + C::BUF(b);
          const uint64_t bo = static_cast<uint64_t>(b * C::DS_TILE) >> 4;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_ss(tb, dK_mn + ((kk * 2048) >> 4), dDS_mn + bo + ((kk * 2048) >> 4), idesc_dq, kk > 0 ? 1u : 0u);
          mma_commit(b_dqfull(b));
        }
      }
      mma_commit(b_done);
      mma_commit(b_drain(role));
      wait_bar(b_drain(role), 0, p.timeout_ns, abort_flag, WB_DRAIN);
    }
    __syncwarp();
  } else if (warp < 8) {
    // ------------------------------------------------------------ elementwise: P^T, dS^T
    const int g = warp >> 2;        // column group: queries 32g .. 32g+31 of the tile
    const int k = threadIdx.x & 127;  // key within the tile == TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const float sl2 = p.scale_log2;
    bool ok = true;
    for (int it = 0; it < n_it; ++it) {
      const int b = it & 1, s = it % NS;
      if (!__all_sync(0xffffffffu, wait_bar(b_sdp(b), (it >> 1) & 1, p.timeout_ns, abort_flag, WB_SDP))) {
        ok = false;
        break;
      }
      // LSE/D of this stage were landed by the producer on q_full[s]; acquire them here too.
      if (!__all_sync(0xffffffffu, wait_bar(b_qfull(s), (it / NS) & 1, p.timeout_ns, abort_flag, WB_QF))) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t tS = tmem + lane_off + C::BUF(b), tDP = tS + 64;
      const float4* lse4 = reinterpret_cast<const float4*>(smem + C::OFF_LSE + s * BQ * 4) + 8 * g;
      const float4* dd4 = reinterpret_cast<const float4*>(smem + C::OFF_DD + s * BQ * 4) + 8 * g;
      const int q0 = (it0 + it) * BQ + 32 * g;  // first query of this group's columns
      const bool need_mask = CAUSAL && (q0 < key0 + 127);
      const int kq = key0 + k - q0;  // masked where column c < kq (key > query)
      uint32_t u[32], w[32];
      tmem_ld32_pair(tS + 32 * g, tDP + 32 * g, u, w);  // S^T and dP^T columns in one round trip
      float pv[32];
#pragma unroll
      for (int c4 = 0; c4 < 8; ++c4) {
        const float4 l = lse4[c4];
        pv[4 * c4 + 0] = ex2_approx(fmaf(__uint_as_float(u[4 * c4 + 0]), sl2, -l.x));
        pv[4 * c4 + 1] = ex2_approx(fmaf(__uint_as_float(u[4 * c4 + 1]), sl2, -l.y));
        pv[4 * c4 + 2] = ex2_approx(fmaf(__uint_as_float(u[4 * c4 + 2]), sl2, -l.z));
        pv[4 * c4 + 3] = ex2_approx(fmaf(__uint_as_float(u[4 * c4 + 3]), sl2, -l.w));
      }
      if (need_mask) {
#pragma unroll
        for (int c = 0; c < 32; ++c) pv[c] = (c < kq) ? 0.f : pv[c];
      }
      uint32_t pk[16];
#pragma unroll
      for (int c = 0; c < 16; ++c) pk[c] = bpack2<BF16>(pv[2 * c], pv[2 * c + 1]);
      // Each group packs into the first half of its own 32 columns, never into columns the other
      // group may still be reading: queries 32g + 2c, 2c+1 go to column 32g + c.
      tmem_st16(tS + 32 * g, pk);
#pragma unroll
      for (int c4 = 0; c4 < 8; ++c4) {
        const float4 dd = dd4[c4];
        pk[2 * c4] = bpack2<BF16>(pv[4 * c4] * (__uint_as_float(w[4 * c4]) - dd.x),
                                  pv[4 * c4 + 1] * (__uint_as_float(w[4 * c4 + 1]) - dd.y));
        pk[2 * c4 + 1] = bpack2<BF16>(pv[4 * c4 + 2] * (__uint_as_float(w[4 * c4 + 2]) - dd.z),
                                      pv[4 * c4 + 3] * (__uint_as_float(w[4 * c4 + 3]) - dd.w));
      }
      tmem_st16(tDP + 32 * g, pk);
      // dS^T row k, queries 32g .. 32g+31: 16-byte units 4g .. 4g+3 of the 128-byte swizzled row
      uint8_t* row = smem + C::OFF_DS + b * C::DS_TILE + k * 128;
#pragma unroll
      for (int u4 = 0; u4 < 4; ++u4)
        *reinterpret_cast<uint4*>(row + (((4 * g + u4) ^ (k & 7)) << 4)) =
            make_uint4(pk[4 * u4], pk[4 * u4 + 1], pk[4 * u4 + 2], pk[4 * u4 + 3]);
      fence_proxy_async_smem();
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(b_ds(b));
    }
    if (g == 0) {
      if (ok) ok = __all_sync(0xffffffffu, wait_bar(b_done, 0, p.timeout_ns, abort_flag, WB_DONE));
      if (ok) tc_fence_after();
      bwd_store_acc<D, BF16>(tmem + lane_off + C::DV_COL, smem + C::OFF_Q, &p.tm_dv, row_base + key0, k, 1.0f, 1, ok,
                             abort_flag);
    }
  } else if (warp < 12) {
    // ------------------------------------------------------------ dQ read-out, then dK epilogue
    const int t = threadIdx.x - 256;  // TMEM lane = d index of dQ^T
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
        tmem_ld32_pair(tmem + lane_off + C::BUF(b), tmem + lane_off + C::BUF(b) + 32, u0, u1);
        tc_fence_before();
        mbar_arrive(b_dqfree(b));
      } else {
#pragma unroll
        for (int c = 0; c < 32; ++c) u0[c] = u1[c] = 0u;
      }
      // the single staging buffer is free once the previous reduce has read it
      if (t == 0) bulk_wait_read0();
      named_bar_sync(2, 128);
      float* st = reinterpret_cast<float*>(smem + C::OFF_DQ);
#pragma unroll
      for (int c = 0; c < 32; ++c) {  // lane t = d index; column c = query
        st[c * D + t] = __uint_as_float(u0[c]);
        st[(32 + c) * D + t] = __uint_as_float(u1[c]);
      }
      fence_proxy_async_smem();
      named_bar_sync(2, 128);
      if (t == 0 && ok && *abort_flag == 0u) {
        bulk_reduce_add_f32(p.dqacc + static_cast<size_t>(row_base + (it0 + it) * BQ) * D, sDQ, C::DQ_STAGE);
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
  if (warp == 13) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace fa
