// Attention backward main kernel for d = 256 (K3, head-dimension split).
//
// Method and per-step arithmetic as fa_bwd_main_kernel (page
// "transformer模型详解（十）：FlashAttention优化技术", section "Re-computation 而非缓存":
// outer loop over K/V column blocks, inner loop over Q row blocks, P rebuilt from
// the saved LSE). What d = 256 changes is the memory plan: the fp32 accumulators
// dV and dK of a 128-key block are 256 tensor-memory columns each, all of TMEM.
// So a CTA makes two passes over its query tiles, one per half h of the head
// dimension. Each pass recomputes
//   S^T = K Q^T and dP^T = V dO^T          (contracted over the full d = 256),
//   P = exp2(S^T * scale * log2 e - LSE * log2 e),  dS = P (dP - D),
// and accumulates only that pass's half of the outputs:
//   dV[:, h] += P^T dO[:, h],  dK[:, h] += dS^T Q[:, h],  dQ[:, h] += dS K[:, h].
// S^T and dP^T are computed twice, so the kernel does 1.4x the useful FLOPs.
// Shared memory: K and V of the block stay resident (128 KB); Q and dO of one
// 64-query step (64 KB) and dS^T (16 KB) complete it, with no room for a second
// stage. The stage is therefore released in two halves of the head dimension:
// the half a pass does not accumulate (chunks 2(1-h), 2(1-h)+1 of Q and dO) is
// read only by S^T and dP^T, so the next step's copy of it is loaded while this
// step's P, dS, dV, dK and dQ^T are formed; the pass's own half, read by dV and
// dK as well, is reloaded once those have completed. S^T and dP^T of a step
// contract over the early half first. LSE and D are double-buffered, each
// buffer released by the elementwise warps.
// dQ^T of a step goes from TMEM straight to the fp32 accumulator with coalesced
// global reductions (a warp covers 128 contiguous bytes per query), and the
// dV/dK epilogue of a pass is staged in the Q and dO tiles.
// TMEM: S^T at 0, dP^T at 64, dQ^T at 128, dV half at 256, dK half at 384. Each
// elementwise group packs P^T (dS^T) of its 32 queries into the first 16 of its
// own 32 columns of S^T (dP^T), never into columns the other group may still be
// reading, so the 16-query slices of the TMEM operand sit at 0, 8, 32, 40.
// Roles (512 threads): warps 0-7 elementwise (two groups of 32 query columns)
// and the dV epilogue (one half of the columns each), warps 8-11 dQ read-out
// and the dK epilogue, warp 12 TMA producer, warps 13-15 MMA issuers: S^T and
// dV (13), dP^T and dK (14), dQ^T (15). One thread issues an MMA only
// every ~100 cycles, so a single issuer could not keep the tensor core busy
// with the 48 products of a step. Each issuer overwrites a TMEM buffer only
// after its own earlier products that read it (MMAs of one thread execute in
// order); the elementwise warps write dS^T(g) to shared memory only once
// dQ^T(g - 1), which reads it, has completed.
#pragma once
#include "fa_bwd_main.cuh"
#include "fa_bwd_order.cuh"

namespace fa {

// L2 prefetch of one box of a 3-D tensor map: nothing is written to shared memory and no
// barrier is signalled (x follows the same 16-byte rule as a load).
__device__ __forceinline__ void tma_prefetch_l2_3d(const void* map, int x, int y, int z) {
  asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(map), "r"(x), "r"(y),
               "r"(z)
               : "memory");
}

struct BwdD256Cfg {
  static constexpr int D = 256, DH = 128, BK = 128, BQ = 64, NCH = D / 64;
  static constexpr int KV_CHUNK = BK * 128;    // 16 KB: 128 rows x 64 elements
  static constexpr int KV_TILE = BK * D * 2;   // 64 KB
  static constexpr int Q_CHUNK = BQ * 128;     // 8 KB: 64 rows x 64 elements
  static constexpr int Q_TILE = BQ * D * 2;    // 32 KB
  static constexpr int DS_TILE = BK * BQ * 2;  // 16 KB: dS^T [128 keys][64 queries]
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = OFF_K + KV_TILE;
  static constexpr int OFF_Q = OFF_V + KV_TILE;
  static constexpr int OFF_DO = OFF_Q + Q_TILE;
  static constexpr int OFF_DS = OFF_DO + Q_TILE;
  static constexpr int OFF_LSE = OFF_DS + DS_TILE;  // two buffers of BQ floats
  static constexpr int OFF_DD = OFF_LSE + 2 * BQ * 4;
  static constexpr int OFF_BAR = OFF_DD + 2 * BQ * 4;
  // bars: kv, q_full / q_empty of the early half (x) and of the pass's own half (w), sdp, ds, dq_full,
  // dq_free, done, epi, drain, lse_full[2], lse_empty[2]
  static constexpr int NBAR = 16;
  static constexpr int SMEM_BYTES = 1024 + OFF_BAR + NBAR * 8 + 16;
  static constexpr int THREADS = 512;
  static constexpr int W_RO = 8, W_PROD = 12, W_ISS = 13;  // first warp of each role after the elementwise
  static constexpr uint32_t S_COL = 0, DP_COL = 64, DQ_COL = 128, DV_COL = 256, DK_COL = 384;
  static_assert(SMEM_BYTES <= 232448, "smem budget");
  static_assert(Q_TILE >= BK * DH * 2, "a pass's dV or dK half (bf16) is staged in the Q or dO tile");
};

template <bool BF16, bool CAUSAL>
__global__ void __launch_bounds__(512, 1) fa_bwd_d256_kernel(const __grid_constant__ BwdParams p) {
  using C = BwdD256Cfg;
  constexpr int BQ = C::BQ, D = C::D, DH = C::DH;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t s0 = smem_u32(smem);
  const uint32_t sK = s0 + C::OFF_K, sV = s0 + C::OFF_V, sQ = s0 + C::OFF_Q, sDO = s0 + C::OFF_DO;
  const uint32_t sDS = s0 + C::OFF_DS;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  const uint32_t b_kv = smem_u32(&bars[0]);
  const uint32_t b_qfx = smem_u32(&bars[1]);
  const uint32_t b_qex = smem_u32(&bars[2]);
  const uint32_t b_sdp = smem_u32(&bars[3]);
  const uint32_t b_ds = smem_u32(&bars[4]);
  const uint32_t b_dqfull = smem_u32(&bars[5]);
  const uint32_t b_dqfree = smem_u32(&bars[6]);
  const uint32_t b_done = smem_u32(&bars[7]);
  const uint32_t b_epi = smem_u32(&bars[8]);
  const uint32_t b_drain = smem_u32(&bars[9]);
  const uint32_t b_qfw = smem_u32(&bars[10]);
  const uint32_t b_qew = smem_u32(&bars[11]);
  const uint32_t b_lfull0 = smem_u32(&bars[12]);   // + 8 * buffer
  const uint32_t b_lempty0 = smem_u32(&bars[14]);  // + 8 * buffer
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(&bars[C::NBAR]);
  volatile uint32_t* abort_flag = tmem_slot + 1;

  const int warp = threadIdx.x >> 5;
  const int N = p.N;
  int bh, kb;  // K/V head (b, h_kv) and key block: see fa_bwd_order.cuh
  bwd_block_order(blockIdx.x, blockIdx.y, gridDim.x, gridDim.y, static_cast<long long>(p.H / p.Hkv) * N * 8ll * D, bh,
                  kb);
  const int key0 = kb * 128;
  const BwdGroup<true> grp(bh, p);  // the query heads that share this K/V head, and the batch's key count
  const int it0 = CAUSAL ? (key0 / BQ) : 0;
  const int n_ith = (N + BQ - 1) / BQ - it0;  // query steps per query head (the last may run past N: masked)
  const int n_it = grp.G * n_ith;             // query steps per pass, head by head
  const int n_g = 2 * n_it;                   // steps of both passes: g = h * n_it + it

  if (threadIdx.x == 0) {
    mbar_init(b_kv, 1);
    mbar_init(b_qfx, 1);
    mbar_init(b_qex, 2);  // S^T and dP^T issuers
    mbar_init(b_qfw, 1);
    mbar_init(b_qew, 2);  // dV and dK
    for (int i = 0; i < 2; ++i) {
      mbar_init(b_lfull0 + 8 * i, 1);
      mbar_init(b_lempty0 + 8 * i, 256);
    }
    mbar_init(b_sdp, 2);
    mbar_init(b_ds, 256);
    mbar_init(b_dqfull, 1);
    mbar_init(b_dqfree, 128);
    mbar_init(b_done, 2);
    mbar_init(b_epi, 3);  // one thread of each epilogue group (two dV halves, dK), once per pass
    mbar_init(b_drain, 3);
    *abort_flag = 0u;
    mbar_fence_init();
    fence_proxy_async_smem();
  }
  if (warp == C::W_ISS) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == C::W_PROD) {
    // ------------------------------------------------------------ producer
    if (elect_one()) {
      tma_prefetch_desc(&p.tm_q);
      tma_prefetch_desc(&p.tm_do);
      mbar_arrive_expect_tx(b_kv, 2 * C::KV_TILE);
#pragma unroll
      for (int c = 0; c < C::NCH; ++c) {
        tma_load_3d(sK + c * C::KV_CHUNK, &p.tm_k, b_kv, c * 64, key0, bh);
        tma_load_3d(sV + c * C::KV_CHUNK, &p.tm_v, b_kv, c * 64, key0, bh);
      }
      int n_x = 0, n_w = 0, n_l = 0;  // copies issued on q_full x, q_full w and the LSE/D buffers
      for (int g = 0; g < n_g; ++g) {
        const int h = g / n_it, it = g % n_it;
        const int cw = 2 * h, cx = 2 - 2 * h;  // first chunk of the pass's own half, of the early half
        // the early half of step g - 1 is free once its S^T and dP^T have completed; the first step of
        // the second pass waits for the first pass's epilogue instead, which staged dV / dK in Q and dO
        if (g == n_it) {
          if (!wait_bar(b_epi, 0, p.timeout_ns, abort_flag, WB_QE)) break;
        } else if (g > 0 && !wait_bar(b_qex, (g - 1) & 1, p.timeout_ns, abort_flag, WB_QE)) {
          break;
        }
        int qh, qs;
        grp.step(it, it0, n_ith, qh, qs);
        const int q_in = qs * BQ;             // within query head qh; rows past N arrive as zeros
        const int qrow = qh * p.Npad + q_in;  // LSE*log2e / D past N: the head's zero padding, masked
        // LSE / D into buffer g & 1 once the elementwise warps have read step g - 2's
        const int lb = g & 1;
        if (g >= 2 && !wait_bar(b_lempty0 + 8 * lb, ((g >> 1) - 1) & 1, p.timeout_ns, abort_flag, WB_QE)) break;
        mbar_arrive_expect_tx(b_lfull0 + 8 * lb, 2 * BQ * 4);
        bulk_load(s0 + C::OFF_LSE + lb * BQ * 4, p.lse2 + qrow, BQ * 4, b_lfull0 + 8 * lb);
        bulk_load(s0 + C::OFF_DD + lb * BQ * 4, p.Dvec + qrow, BQ * 4, b_lfull0 + 8 * lb);
        ++n_l;
        mbar_arrive_expect_tx(b_qfx, C::Q_TILE);  // two chunks of Q and two of dO
#pragma unroll
        for (int c = cx; c < cx + 2; ++c) {
          tma_load_3d(sQ + c * C::Q_CHUNK, &p.tm_q, b_qfx, c * 64, q_in, qh);
          tma_load_3d(sDO + c * C::Q_CHUNK, &p.tm_do, b_qfx, c * 64, q_in, qh);
        }
        ++n_x;
        // the pass's own half of step g - 1 is free once dV and dK have read it
        if (g != n_it && g > 0 && !wait_bar(b_qew, (g - 1) & 1, p.timeout_ns, abort_flag, WB_QE)) break;
        mbar_arrive_expect_tx(b_qfw, C::Q_TILE);
#pragma unroll
        for (int c = cw; c < cw + 2; ++c) {
          tma_load_3d(sQ + c * C::Q_CHUNK, &p.tm_q, b_qfw, c * 64, q_in, qh);
          tma_load_3d(sDO + c * C::Q_CHUNK, &p.tm_do, b_qfw, c * 64, q_in, qh);
        }
        ++n_w;
        // Q and dO of step g + 1 towards L2 now: their loads wait until this step's products release the
        // stage, and then find them in L2 instead of HBM
        if (g + 1 < n_g) {
          int qh1, qs1;
          grp.step((g + 1) % n_it, it0, n_ith, qh1, qs1);
#pragma unroll
          for (int c = 0; c < C::NCH; ++c) {
            tma_prefetch_l2_3d(&p.tm_q, c * 64, qs1 * BQ, qh1);
            tma_prefetch_l2_3d(&p.tm_do, c * 64, qs1 * BQ, qh1);
          }
        }
      }
      // Drain: every issued copy has landed before the CTA may exit.
      wait_bar(b_kv, 0, p.timeout_ns, abort_flag, WB_DRAIN);
      if (n_x > 0) wait_bar(b_qfx, (n_x - 1) & 1, p.timeout_ns, abort_flag, WB_DRAIN);
      if (n_w > 0) wait_bar(b_qfw, (n_w - 1) & 1, p.timeout_ns, abort_flag, WB_DRAIN);
      for (int j = n_l - 2 < 0 ? 0 : n_l - 2; j < n_l; ++j)
        wait_bar(b_lfull0 + 8 * (j & 1), (j >> 1) & 1, p.timeout_ns, abort_flag, WB_DRAIN);
    }
    __syncwarp();
  } else if (warp >= C::W_ISS) {
    // ------------------------------------------------------------ MMA issuers
    const int role = warp - C::W_ISS;  // 0: S^T, dV   1: dP^T, dK   2: dQ^T
    if (elect_one()) {
      constexpr uint32_t idesc_sdp = make_idesc(128, BQ, BF16, false, false);
      constexpr uint32_t idesc_acc = make_idesc(128, DH, BF16, false, true);
      constexpr uint32_t idesc_dq = make_idesc(128, BQ, BF16, true, true);
      // Descriptors are built once; steps add (byte offset >> 4) to the 14-bit start-address
      // field, which cannot carry out of it (shared memory ends below 256 KB).
      // role 0: K and Q (K-major) for S^T, dO (MN-major) for dV; role 1: V and dO for dP^T, Q for dK
      const uint64_t dA_k = make_sdesc(role == 0 ? sK : sV, 16, 1024);
      const uint64_t dB_k = make_sdesc(role == 0 ? sQ : sDO, 16, 1024);
      const uint64_t dB_mn = make_sdesc(role == 0 ? sDO : sQ, C::Q_CHUNK, 1024);
      const uint64_t dKT_mn = make_sdesc(sK, C::KV_CHUNK, 1024);  // K^T as the A operand of dQ^T
      const uint64_t dDS_mn = make_sdesc(sDS, 128 * 128, 1024);   // dS^T as the B operand of dQ^T
      const uint32_t t_sdp = tmem + (role == 0 ? C::S_COL : C::DP_COL);  // S^T or dP^T (then P^T or dS^T)
      const uint32_t t_acc = tmem + (role == 0 ? C::DV_COL : C::DK_COL);
      bool ok = wait_bar(b_kv, 0, p.timeout_ns, abort_flag, WB_KV);
      for (int g = 0; ok && g < n_g; ++g) {
        const int h = g / n_it, it = g % n_it;
        if (role == 2) {
          // dQ^T[h-half][q] = sum_k K[k][h-half] dS^T[k][q]  (M = 128 = half of d, N = 64, K = 128 keys)
          if (!wait_bar(b_ds, g & 1, p.timeout_ns, abort_flag, WB_DS)) break;
          if (g > 0 && !wait_bar(b_dqfree, (g - 1) & 1, p.timeout_ns, abort_flag, WB_DQFREE)) break;
          tc_fence_after();
          const uint64_t half_k = static_cast<uint64_t>((2 * h * C::KV_CHUNK) >> 4);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_ss(tmem + C::DQ_COL, dKT_mn + half_k + ((kk * 2048) >> 4), dDS_mn + ((kk * 2048) >> 4), idesc_dq,
                   kk > 0 ? 1u : 0u);
          mma_commit(b_dqfull);
          continue;
        }
        if (!wait_bar(b_qfx, g & 1, p.timeout_ns, abort_flag, WB_QF)) break;
        // a new pass overwrites the dV / dK halves: the previous pass's epilogue must have read them
        if (g == n_it && !wait_bar(b_epi, 0, p.timeout_ns, abort_flag, WB_DONE)) break;
        tc_fence_after();
        // S^T = K Q^T (role 0) or dP^T = V dO^T (role 1)  (M = 128 keys, N = 64 queries, K = d = 256),
        // contracted over the early half's chunks first, then (once they have landed) the pass's own half
        bool landed = true;
#pragma unroll
        for (int part = 0; part < 2; ++part) {
          if (part == 1) {
            if (!wait_bar(b_qfw, g & 1, p.timeout_ns, abort_flag, WB_QF)) {
              landed = false;
              break;
            }
            tc_fence_after();
          }
          const int c0 = part == 0 ? 2 - 2 * h : 2 * h;
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const int c = c0 + (j >> 2);
            const uint64_t oa = static_cast<uint64_t>((c * C::KV_CHUNK + (j & 3) * 32) >> 4);
            const uint64_t ob = static_cast<uint64_t>((c * C::Q_CHUNK + (j & 3) * 32) >> 4);
            mma_ss(t_sdp, dA_k + oa, dB_k + ob, idesc_sdp, (part > 0 || j > 0) ? 1u : 0u);
          }
        }
        if (!landed) break;
        mma_commit(b_sdp);
        mma_commit(b_qex);  // the early half may be reloaded for step g + 1
        if (!wait_bar(b_ds, g & 1, p.timeout_ns, abort_flag, WB_DS)) break;
        tc_fence_after();
        // dV[:, h] += P^T dO[:, h] (role 0) or dK[:, h] += dS^T Q[:, h] (role 1)
        //   (M = 128 keys, N = 128 = half of d, K = 64 queries; A from TMEM, B MN-major from chunks 2h, 2h+1)
        const uint64_t half_q = static_cast<uint64_t>((2 * h * C::Q_CHUNK) >> 4);
#pragma unroll
        for (int kk = 0; kk < BQ / 16; ++kk)
          mma_ts(t_acc, t_sdp + 32 * (kk >> 1) + 8 * (kk & 1), dB_mn + half_q + ((kk * 2048) >> 4), idesc_acc,
                 (it > 0 || kk > 0) ? 1u : 0u);
        mma_commit(b_qew);  // the pass's own half may be reloaded for step g + 1
        if (it == n_it - 1) mma_commit(b_done);  // this pass's dV / dK halves are final
      }
      mma_commit(b_drain);
      wait_bar(b_drain, 0, p.timeout_ns, abort_flag, WB_DRAIN);
    }
    __syncwarp();
  } else if (warp < C::W_RO) {
    // ------------------------------------------------------------ elementwise: P^T, dS^T; dV epilogue
    const int gq = warp >> 2;            // column group: queries 32 gq .. 32 gq + 31 of the step
    const int k = threadIdx.x & 127;     // key within the tile == TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_off + C::S_COL + 32 * gq, tDP = tmem + lane_off + C::DP_COL + 32 * gq;
    const float sl2 = p.scale_log2;
    bool ok = true;
    for (int g = 0; g < n_g; ++g) {
      const int h = g / n_it, it = g % n_it;
      if (ok && !__all_sync(0xffffffffu, wait_bar(b_sdp, g & 1, p.timeout_ns, abort_flag, WB_SDP))) ok = false;
      // LSE / D of the step, in buffer g & 1 (released below, once read)
      const int lb = g & 1;
      if (ok && !__all_sync(0xffffffffu, wait_bar(b_lfull0 + 8 * lb, (g >> 1) & 1, p.timeout_ns, abort_flag, WB_QF)))
        ok = false;
      if (ok) {
        tc_fence_after();
        const float4* lse4 = reinterpret_cast<const float4*>(smem + C::OFF_LSE + lb * BQ * 4) + 8 * gq;
        const float4* dd4 = reinterpret_cast<const float4*>(smem + C::OFF_DD + lb * BQ * 4) + 8 * gq;
        int qh, qs;
        grp.step(it, it0, n_ith, qh, qs);
        const int q0 = qs * BQ + 32 * gq;  // first query of this group's columns
        // masked: column c < kq (key > query, causal), q0 + c >= N (query past the sequence) or the
        // whole row when the key does not exist (past N or past the batch's key count: S need not
        // come from a real key, and exp(-LSE) need not be finite)
        const bool need_mask = (CAUSAL && (q0 < key0 + 127)) || (q0 + 32 > N) || (key0 + 128 > grp.klen);
        const int kq = CAUSAL ? (key0 + k - q0) : 0;
        const int qn = key0 + k < grp.klen ? N - q0 : 0;
        uint32_t u[32], v[32];
        tmem_ld32_pair(tS, tDP, u, v);  // S^T and dP^T columns in one round trip
        float pv[32];
        // pairs of columns through the two-wide fp32 FMA / add / multiply (each lane rounds as the
        // scalar instruction would)
        const float2 sl2_2 = make_float2(sl2, sl2);
#pragma unroll
        for (int c4 = 0; c4 < 8; ++c4) {
          const float4 l = lse4[c4];
          const float2 x0 = __ffma2_rn(make_float2(__uint_as_float(u[4 * c4 + 0]), __uint_as_float(u[4 * c4 + 1])),
                                       sl2_2, make_float2(-l.x, -l.y));
          const float2 x1 = __ffma2_rn(make_float2(__uint_as_float(u[4 * c4 + 2]), __uint_as_float(u[4 * c4 + 3])),
                                       sl2_2, make_float2(-l.z, -l.w));
          pv[4 * c4 + 0] = ex2_approx(x0.x);
          pv[4 * c4 + 1] = ex2_approx(x0.y);
          pv[4 * c4 + 2] = ex2_approx(x1.x);
          pv[4 * c4 + 3] = ex2_approx(x1.y);
        }
        if (need_mask) {
#pragma unroll
          for (int c = 0; c < 32; ++c) pv[c] = (c < kq || c >= qn) ? 0.f : pv[c];
        }
        uint32_t pk[16];
#pragma unroll
        for (int c = 0; c < 16; ++c) pk[c] = bpack2<BF16>(pv[2 * c], pv[2 * c + 1]);
        tmem_st16(tS, pk);
#pragma unroll
        for (int c4 = 0; c4 < 8; ++c4) {
          const float4 dd = dd4[c4];
          const float2 ds0 = __fmul2_rn(make_float2(pv[4 * c4], pv[4 * c4 + 1]),
                                        __fadd2_rn(make_float2(__uint_as_float(v[4 * c4]), __uint_as_float(v[4 * c4 + 1])),
                                                   make_float2(-dd.x, -dd.y)));
          const float2 ds1 = __fmul2_rn(make_float2(pv[4 * c4 + 2], pv[4 * c4 + 3]),
                                        __fadd2_rn(make_float2(__uint_as_float(v[4 * c4 + 2]),
                                                               __uint_as_float(v[4 * c4 + 3])),
                                                   make_float2(-dd.z, -dd.w)));
          pk[2 * c4] = bpack2<BF16>(ds0.x, ds0.y);
          pk[2 * c4 + 1] = bpack2<BF16>(ds1.x, ds1.y);
        }
        mbar_arrive(b_lempty0 + 8 * lb);  // this thread's last read of the step's LSE / D
        tmem_st16(tDP, pk);
        // dS^T row k, queries 32 gq .. 32 gq + 31: 16-byte units 4 gq .. 4 gq + 3 of the 128-byte swizzled
        // row, over dS^T(g - 1) once dQ^T(g - 1) has read it (a timeout here leaves ok false and the loop
        // running, so the group's epilogue barriers stay uniform)
        if (g == 0 || __all_sync(0xffffffffu, wait_bar(b_dqfull, (g - 1) & 1, p.timeout_ns, abort_flag, WB_DQF))) {
          uint8_t* row = smem + C::OFF_DS + k * 128;
#pragma unroll
          for (int u4 = 0; u4 < 4; ++u4)
            *reinterpret_cast<uint4*>(row + (((4 * gq + u4) ^ (k & 7)) << 4)) =
                make_uint4(pk[4 * u4], pk[4 * u4 + 1], pk[4 * u4 + 2], pk[4 * u4 + 3]);
          fence_proxy_async_smem();
        } else {
          ok = false;
        }
        tmem_st_wait();
        tc_fence_before();
        if (ok) mbar_arrive(b_ds);
      }
      if (it == n_it - 1) {
        // end of pass h: dV[:, h] (128 keys x 128), columns 64 gq .. 64 gq + 63 staged in the Q tile's
        // chunk gq, stored with TMA
        bool ok_e = ok && __all_sync(0xffffffffu, wait_bar(b_done, h & 1, p.timeout_ns, abort_flag, WB_DONE));
        if (ok_e) tc_fence_after();
        bwd_store_acc<64, BF16>(tmem + lane_off + C::DV_COL + 64 * gq, smem + C::OFF_Q + gq * (128 * 128), &p.tm_dv,
                                key0, bh, k, 1.0f, 1 + 2 * gq, ok_e, abort_flag, h * DH + 64 * gq);
        if (k == 0) {
          tc_fence_before();
          mbar_arrive(b_epi);
        }
        ok = ok_e;
      }
    }
  } else {
    // ------------------------------------------------------------ dQ read-out; dK epilogue (warps 8-11)
    const int t = threadIdx.x - 32 * C::W_RO;  // TMEM lane = index within the head-dimension half
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    bool ok = true;
    for (int g = 0; g < n_g; ++g) {
      const int h = g / n_it, it = g % n_it;
      if (ok && !__all_sync(0xffffffffu, wait_bar(b_dqfull, g & 1, p.timeout_ns, abort_flag, WB_DQF))) ok = false;
      if (ok) {
        uint32_t u0[32], u1[32];
        tc_fence_after();
        tmem_ld32(tmem + lane_off + C::DQ_COL, u0);
        tmem_ld32(tmem + lane_off + C::DQ_COL + 32, u1);
        tc_fence_before();
        mbar_arrive(b_dqfree);
        if (*abort_flag == 0u) {
          // dQ[q][h*128 + t] += dQ^T[t][q]: a warp covers 128 contiguous bytes per query
          int qh, qs;
          grp.step(it, it0, n_ith, qh, qs);
          float* dst = p.dqacc + static_cast<size_t>(qh * p.Npad + qs * BQ) * D + h * DH + t;
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            atomicAdd(dst + c * D, __uint_as_float(u0[c]));
            atomicAdd(dst + (32 + c) * D, __uint_as_float(u1[c]));
          }
        }
      }
      if (it == n_it - 1) {
        // end of pass h: dK[:, h] = scale * accumulator, staged in the dO tile
        bool ok_e = ok && __all_sync(0xffffffffu, wait_bar(b_done, h & 1, p.timeout_ns, abort_flag, WB_DONE));
        if (ok_e) tc_fence_after();
        bwd_store_acc<DH, BF16>(tmem + lane_off + C::DK_COL, smem + C::OFF_DO, &p.tm_dk, key0, bh, t, p.scale,
                                2, ok_e, abort_flag, h * DH);
        if (t == 0) {
          tc_fence_before();
          mbar_arrive(b_epi);
        }
        ok = ok_e;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == C::W_ISS) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace fa
