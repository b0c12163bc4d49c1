// Attention backward main kernel for d = 64 and 128 (K3), software-pipelined.
//
// Method (page "transformer模型详解（十）：FlashAttention优化技术", section
// "Re-computation 而非缓存"): outer loop over K/V column blocks, inner loop over Q
// row blocks, P rebuilt from the saved LSE: P = exp(scale * S - LSE),
// dV_j += P^T dO_i, dP = dO_i V_j^T, dS = P * (dP - D_i), dK_j += scale * dS^T Q_i,
// dQ_i += scale * dS K_j. Keys are the MMA's M dimension, so S and dP are
// produced transposed with one key per TMEM lane, and P^T / dS^T feed dV and dK
// straight from TMEM. The schedule keeps the tensor core from waiting for the
// elementwise warps:
//   * S^T and dP^T of query tile i go to one of NB TMEM buffers (i % NB: two for d = 128, three for
//     d = 64, whose smaller accumulators leave the room);
//   * S^T(i+1), dP^T(i+1) are issued into the next buffer *before* the
//     issuers wait for P^T(i), dS^T(i), so the tensor core computes the next
//     scores while the elementwise warps turn the current ones into P and dS;
//   * dQ^T(i) = K^T dS^T(i) is written over S^T(i)'s columns once dV(i) has
//     read P^T(i) from them, and read out before S^T(i+NB) reuses the buffer:
//     each read-out thread holds one row of dQ^T (a d index, 64 queries) and adds
//     it into the fp32 accumulator with global reductions, one coalesced 128-byte
//     row segment per warp instruction (a shared staging tile drained by bulk
//     reductions measured 6% slower at d = 64 and no faster at d = 128);
//   * dS^T goes to one of NB shared-memory tiles (the dQ operand), and
//     Q, dO, LSE*log2e, D stream through a three-stage TMA ring;
//   * for d = 64, dQ^T = K^T dS^T still has M = 128: a zeroed chunk after K
//     pads K^T with 64 zero rows, whose dQ^T lanes are never read.
// TMEM (512 columns): buffer b at 128b holds S^T/P^T (cols 0-63, then dQ^T)
// and dP^T/dS^T (cols 64-127); dV at 128 NB, dK after it (d columns each). Packed
// 16-bit P^T of queries 32g..32g+31 sits in columns 32g..32g+15 (dS^T likewise
// from 64).
// Roles (16 warps, 4 per SM sub-partition): warps 0-7 elementwise, in two
// groups that each own 32 of the tile's 64 query columns; warps 8-11 dQ
// read-out and the dK epilogue; warp 12 TMA producer; warps 13-15 MMA issuers
// (S^T + dV, dP^T + dK, dQ^T), since one thread cannot issue fast enough.
// DQACC = false is the kernel for the separate dQ pass (fa_bwd_dq.cuh): it
// computes dK and dV only, so no dQ^T product, no dS^T tile in shared memory and
// no read-out; a buffer is then refilled as soon as the same issuer's dV / dK of
// NB steps before (issued earlier by that thread, executed in order) have read it.
// Key blocks run in the L2-grouped launch order of fa_bwd_order.cuh.
#pragma once
#include "fa_bwd_main.cuh"
#include "fa_bwd_order.cuh"

namespace fa {

template <int D_>
struct BwdPipeCfg {
  static constexpr int D = D_, BK = 128, BQ = 64, NCH = D / 64, NSTAGE = 3;
  // TMEM buffers for S^T/dP^T (then dQ^T) of consecutive query steps: step g uses buffer g % NB. With
  // d = 64 the dV and dK accumulators take 64 columns each, which leaves room for a third buffer.
  static constexpr int NB = D < 128 ? 3 : 2;
  static constexpr int KV_CHUNK = BK * 128;   // 16 KB: 128 rows x 128 bytes (64 elements)
  static constexpr int KV_TILE = BK * D * 2;  // 32 KB (d = 128), 16 KB (d = 64)
  // dQ^T = K^T dS^T needs M = 128 rows of K^T: for d = 64 a zeroed chunk follows K, so the MMA
  // sees K^T padded with 64 zero rows (those dQ^T lanes are never read)
  static constexpr int K_REGION = (D < 128 ? 2 : NCH) * KV_CHUNK;
  static constexpr int Q_CHUNK = BQ * 128;    // 8 KB
  static constexpr int Q_TILE = BQ * D * 2;   // 16 KB (d = 128), 8 KB (d = 64)
  static constexpr int DS_TILE = BK * BQ * 2;  // 16 KB: dS^T [128 keys][64 queries]
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = OFF_K + K_REGION;
  static constexpr int OFF_Q = OFF_V + KV_TILE;             // NSTAGE stages
  static constexpr int OFF_DO = OFF_Q + NSTAGE * Q_TILE;    // NSTAGE stages
  static constexpr int OFF_DS = OFF_DO + NSTAGE * Q_TILE;   // NB buffers
  static constexpr int OFF_LSE = OFF_DS + NB * DS_TILE;     // NSTAGE x BQ floats
  static constexpr int OFF_DD = OFF_LSE + NSTAGE * BQ * 4;  // NSTAGE x BQ floats
  static constexpr int OFF_BAR = OFF_DD + NSTAGE * BQ * 4;
  // bars: kv, q_full[3], q_empty[3], sdp[NB], ds[NB], dq_full[NB], dq_free[NB], dv_done[NB], done, drain[3],
  // v_free, k_free, clc, item_full[2], item_empty[2]
  static constexpr int NBAR = 1 + 2 * NSTAGE + 5 * NB + 1 + 3 + 2 + 1 + 4;
  static constexpr int BAR_BYTES = (NBAR * 8 + 15) & ~15;
  // after the barriers: the 16-byte launch-control answer, the item queue (2 x {x, y}), TMEM slot + abort flag
  static constexpr int SMEM_BYTES = 1024 + OFF_BAR + BAR_BYTES + 16 + 16 + 16;
  static constexpr int THREADS = 512;
  // Register split: launched at LAUNCH_REGS a thread (four warps per SM sub-partition); the
  // elementwise warpgroups then take EW_REGS from the producer / MMA warpgroup (OTHER_REGS); the
  // read-out warpgroup keeps the launch count. The host refuses to launch unless the compiled count
  // equals LAUNCH_REGS, so the increase always finds its registers.
  static constexpr int LAUNCH_REGS = 128, EW_REGS = 136, OTHER_REGS = 112;
  static_assert(128 * (2 * EW_REGS + LAUNCH_REGS + OTHER_REGS) <= THREADS * LAUNCH_REGS, "register split");
  static constexpr int ITEM_READERS = 3 + 8 + 1;  // the MMA threads, one lane per elementwise warp, read-out thread 0
  __host__ __device__ static constexpr uint32_t BUF(int b) { return 128u * b; }
  static constexpr uint32_t DV_COL = 128u * NB, DK_COL = DV_COL + D;
  static_assert(DK_COL + D <= 512, "TMEM budget");
  static_assert(D == 64 || D == 128, "d = 64 or 128");
  static_assert(SMEM_BYTES <= 232448, "smem budget");
};

// The K/V head and key block that launch index (x, y) works on (fa_bwd_order.cuh).
struct BwdSlot {
  int bh, kb;
  __device__ __forceinline__ BwdSlot(int x, int y, const BwdParams& p, int d) {
    bwd_block_order(x, y, gridDim.x, gridDim.y, static_cast<long long>(p.H / p.Hkv) * p.N * 8ll * d, bh, kb);
  }
};

// One work item: the 128-key block of a K/V head that the CTA launched as (x, y) stands for (the
// launch order takes heads in L2-sized groups, longest blocks first within a group; under causal
// masking block 0 has the most query steps). The block's query steps run over the G query heads
// that share the K/V head, one head after another.
template <bool CAUSAL, bool GRP>
struct BwdItem {
  BwdSlot slot;
  int bh;        // K/V head (b, h_kv): the z coordinate of the K, V maps
  int row_base;  // row of (b, h_kv, 0) in the [B*Hkv*N, d] view of K, V, dK, dV
  int key0;      // first key of the block
  int it0;       // first 64-query step of each query head (causal: the block's diagonal)
  int n_ith;     // query steps per query head (the last may run past N: its extra queries are masked)
  int n_it;      // query steps of the block: G * n_ith
  BwdGroup<GRP> grp;  // the query heads of the group and the batch's key count
  __device__ __forceinline__ BwdItem(int x, int y, const BwdParams& p, int d) : slot(x, y, p, d), grp(slot.bh, p) {
    bh = slot.bh;
    row_base = bh * p.N;
    key0 = slot.kb * 128;
    it0 = CAUSAL ? (key0 / 64) : 0;  // 64-query steps
    n_ith = (p.N + 63) / 64 - it0;
    n_it = grp.G * n_ith;
  }
};

// GRP: grouped K/V heads or a key-padding mask (the general form); false for plain multi-head attention.
// DQACC: dQ partials accumulated here (true) or left to the separate dQ pass (false).
template <int D_, bool BF16, bool CAUSAL, bool GRP, bool DQACC>
__global__ void __launch_bounds__(512, 1) fa_bwd_pipe_kernel(const __grid_constant__ BwdParams p) {
  using C = BwdPipeCfg<D_>;
  using Item = BwdItem<CAUSAL, GRP>;
  constexpr int BQ = C::BQ, D = C::D, NS = C::NSTAGE;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t s0 = smem_u32(smem);
  const uint32_t sK = s0 + C::OFF_K, sV = s0 + C::OFF_V, sQ = s0 + C::OFF_Q, sDO = s0 + C::OFF_DO;
  const uint32_t sDS = s0 + C::OFF_DS;
  uint8_t* aux = smem + C::OFF_BAR;
  uint64_t* bars = reinterpret_cast<uint64_t*>(aux);
  const uint32_t b_kv = smem_u32(&bars[0]);
  auto b_qfull = [&](int s) { return smem_u32(&bars[1 + s]); };
  auto b_qempty = [&](int s) { return smem_u32(&bars[1 + NS + s]); };
  constexpr int NB = C::NB, B0 = 1 + 2 * NS, B1 = B0 + 5 * NB;  // first per-buffer bar, first bar after them
  auto b_sdp = [&](int b) { return smem_u32(&bars[B0 + b]); };
  auto b_ds = [&](int b) { return smem_u32(&bars[B0 + NB + b]); };
  auto b_dqfull = [&](int b) { return smem_u32(&bars[B0 + 2 * NB + b]); };
  auto b_dqfree = [&](int b) { return smem_u32(&bars[B0 + 3 * NB + b]); };
  auto b_dvdone = [&](int b) { return smem_u32(&bars[B0 + 4 * NB + b]); };
  const uint32_t b_done = smem_u32(&bars[B1]);
  auto b_drain = [&](int i) { return smem_u32(&bars[B1 + 1 + i]); };
  const uint32_t b_vfree = smem_u32(&bars[B1 + 4]);
  const uint32_t b_kfree = smem_u32(&bars[B1 + 5]);
  const uint32_t b_clc = smem_u32(&bars[B1 + 6]);
  auto b_item_full = [&](int i) { return smem_u32(&bars[B1 + 7 + i]); };
  auto b_item_empty = [&](int i) { return smem_u32(&bars[B1 + 9 + i]); };
  const uint32_t clc_resp = smem_u32(aux + C::BAR_BYTES);
  volatile int* items = reinterpret_cast<volatile int*>(aux + C::BAR_BYTES + 16);  // [2][2]: x, y (x < 0: none)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(aux + C::BAR_BYTES + 32);
  volatile uint32_t* abort_flag = tmem_slot + 1;
  volatile int* dq_next = reinterpret_cast<volatile int*>(tmem_slot + 2);  // read-out group's copy of {x, y}

  const int warp = threadIdx.x >> 5;
  const int N = p.N;

  if (threadIdx.x == 0) {
    mbar_init(b_kv, 1);
    for (int s = 0; s < NS; ++s) {
      mbar_init(b_qfull(s), 1);
      mbar_init(b_qempty(s), 2);  // released by issuers A (after dV) and B (after dK)
    }
    for (int b = 0; b < NB; ++b) {
      mbar_init(b_sdp(b), 2);  // S^T from issuer A, dP^T from issuer B
      mbar_init(b_ds(b), 256);
      mbar_init(b_dqfull(b), 1);
      mbar_init(b_dqfree(b), 128);
      mbar_init(b_dvdone(b), 1);
    }
    mbar_init(b_done, 3);
    for (int i = 0; i < 3; ++i) mbar_init(b_drain(i), 1);
    mbar_init(b_vfree, 256);
    mbar_init(b_kfree, 128);
    mbar_init(b_clc, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(b_item_full(i), 1);
      mbar_init(b_item_empty(i), C::ITEM_READERS);
    }
    *abort_flag = 0u;
    mbar_fence_init();
    fence_proxy_async_smem();
  }
  if (warp == 13) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  if constexpr (D < 128) {
    // the zero rows that pad K^T to M = 128 for dQ^T; never overwritten
    uint4* z = reinterpret_cast<uint4*>(smem + C::OFF_K + C::KV_CHUNK);
    for (int i = threadIdx.x; i < C::KV_CHUNK / 16; i += C::THREADS) z[i] = make_uint4(0u, 0u, 0u, 0u);
    fence_proxy_async_smem();  // visible to the tensor core (async proxy)
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // Work loop shared by all roles (as in the forward): the CTA starts with the key block it was
  // launched for; the producer takes over not-yet-launched CTAs (cluster launch control, asked
  // two query steps before the end of the current block) and passes their ids through a
  // two-entry queue; an id x < 0 ends the loop. Barrier phases run on per-role step and block
  // counters, so nothing is re-initialised between blocks. The next block's K and V overwrite
  // the current ones once every MMA of the current block has completed (done); its first query
  // stages are loaded before that. dV and dK are read out of TMEM at the end of a block
  // (v_free, k_free release the accumulators to the next block) and stored from registers.
  // Reads the queue entry that names the block after block index `n` (the MMA threads and one
  // lane of each elementwise / read-out warp read it; the caller has already synchronised its warp).
  auto next_item = [&](int n, bool arrive, int& x, int& y) -> bool {
    if (!wait_bar(b_item_full(n & 1), (n >> 1) & 1, p.timeout_ns, abort_flag, WB_ITEM)) return false;
    x = items[2 * (n & 1)];
    y = items[2 * (n & 1) + 1];
    if (arrive) mbar_arrive(b_item_empty(n & 1));
    return x >= 0;
  };

  // Each role changes its register budget (the read-out warpgroup keeps it) and ends with its own
  // copy of the teardown barrier, so no code is shared between two budgets.
  if (warp == 12) {
    // ------------------------------------------------------------ producer
    setmaxnreg_dec<C::OTHER_REGS>();
    if (elect_one()) {
      tma_prefetch_desc(&p.tm_q);
      tma_prefetch_desc(&p.tm_do);
      tma_prefetch_desc(&p.tm_k);
      tma_prefetch_desc(&p.tm_v);
      int ix = blockIdx.x, iy = blockIdx.y;
      uint32_t gs = 0;  // query stages issued (all blocks)
      int nb = 0;       // blocks whose K/V were issued
      bool clc_live = true, clc_pending = false, ok = true;
      uint32_t clc_phase = 0;
      auto load_stage = [&](const Item& w, int it) -> bool {
        const uint32_t s = gs % NS, use = gs / NS;
        if (use > 0 && !wait_bar(b_qempty(s), (use - 1) & 1, p.timeout_ns, abort_flag, WB_QE)) return false;
        int qh, qs;
        w.grp.step(it, w.it0, w.n_ith, qh, qs);
        const int q_in = qs * BQ;  // first query of the step within query head qh
        const int qrow = qh * p.Npad + q_in;
        mbar_arrive_expect_tx(b_qfull(s), 2 * C::Q_TILE + 2 * BQ * 4);
#pragma unroll
        for (int c = 0; c < C::NCH; ++c) {
          tma_load_3d(sQ + s * C::Q_TILE + c * C::Q_CHUNK, &p.tm_q, b_qfull(s), c * 64, q_in, qh);
          tma_load_3d(sDO + s * C::Q_TILE + c * C::Q_CHUNK, &p.tm_do, b_qfull(s), c * 64, q_in, qh);
        }
        // LSE*log2e and D rows past N (a step that runs past the sequence) are the head's padding
        // rows (zeros), and the queries they belong to are masked
        bulk_load(s0 + C::OFF_LSE + s * BQ * 4, p.lse2 + qrow, BQ * 4, b_qfull(s));
        bulk_load(s0 + C::OFF_DD + s * BQ * 4, p.Dvec + qrow, BQ * 4, b_qfull(s));
        ++gs;
        return true;
      };
      auto ask = [&]() {
        if (!clc_live) return;
        fence_proxy_async_smem();  // earlier generic reads of the answer slot come first
        mbar_arrive_expect_tx(b_clc, 16);
        clc_try_cancel(clc_resp, b_clc);
        clc_pending = true;
      };
      while (ok) {
        const Item w(ix, iy, p, D);
        const int pre = w.n_it < 2 ? w.n_it : 2;  // stages issued before the block's K/V can be
        const int ask_at = w.n_it - 2 > 0 ? w.n_it - 2 : 0;
        int it = 0;
        for (; ok && it < pre; ++it) ok = load_stage(w, it);
        if (!ok) break;
        // K and V of the previous block are dead once all of its MMAs have completed
        if (nb > 0 && !wait_bar(b_done, (nb - 1) & 1, p.timeout_ns, abort_flag, WB_DONE)) break;
        mbar_arrive_expect_tx(b_kv, 2 * C::KV_TILE);
#pragma unroll
        for (int c = 0; c < C::NCH; ++c) {
          tma_load_3d(sK + c * C::KV_CHUNK, &p.tm_k, b_kv, c * 64, w.key0, w.bh);
          tma_load_3d(sV + c * C::KV_CHUNK, &p.tm_v, b_kv, c * 64, w.key0, w.bh);
        }
        ++nb;
        if (ask_at < pre) ask();
        for (; ok && it < w.n_it; ++it) {
          if (it == ask_at) ask();
          ok = load_stage(w, it);
        }
        if (!ok) break;
        int nx = -1, ny = 0;
        if (clc_live) {
          if (!wait_bar(b_clc, clc_phase, p.timeout_ns, abort_flag, WB_CLC)) break;
          clc_pending = false;
          clc_phase ^= 1u;
          if (!clc_query(clc_resp, nx, ny)) {
            clc_live = false;
            nx = -1;
          } else if (nx < 0 || ny < 0 || nx >= static_cast<int>(gridDim.x) || ny >= static_cast<int>(gridDim.y)) {
            report_status(FA_DEV_BAD_INDEX, WB_CLC);  // a taken-over CTA must be one of this grid's
            clc_live = false;
            nx = -1;
          }
        }
        const int qi = nb - 1;  // queue entry qi names the block after block qi
        if (qi >= 2 && !wait_bar(b_item_empty(qi & 1), ((qi >> 1) - 1) & 1, p.timeout_ns, abort_flag, WB_ITEM))
          break;
        items[2 * (qi & 1)] = nx;
        items[2 * (qi & 1) + 1] = ny;
        mbar_arrive(b_item_full(qi & 1));  // release: readers acquire through their wait
        if (nx < 0) break;
        ix = nx;
        iy = ny;
      }
      // Drain: every issued copy has landed before the CTA may exit.
      if (clc_pending) wait_bar(b_clc, clc_phase, p.timeout_ns, abort_flag, WB_DRAIN);
      if (nb > 0) wait_bar(b_kv, (nb - 1) & 1, p.timeout_ns, abort_flag, WB_DRAIN);
      for (uint32_t g = (gs > NS ? gs - NS : 0u); g < gs; ++g)
        wait_bar(b_qfull(g % NS), (g / NS) & 1, p.timeout_ns, abort_flag, WB_DRAIN);
    }
    __syncwarp();
    tc_fence_before();
    __syncthreads();
  } else if (warp >= 13) {
    // ------------------------------------------------------------ MMA issuers
    // One thread issues a tcgen05.mma only every ~100+ cycles, so the step's 32 MMAs are spread
    // over three warps: A = S^T and dV, B = dP^T and dK, C = dQ^T. A's and B's accumulators are
    // disjoint; C writes dQ^T over the S^T/P^T columns of the step, so it first waits for dV
    // (issuer A) to have read P^T there (dv_done). A only re-fills a buffer after warps 8-11 have
    // read the dQ^T that C left in it (dq_free). The first dV / dK MMA of a block overwrites the
    // accumulator, so it waits until the previous block's epilogue has read it (v_free / k_free).
    setmaxnreg_dec<C::OTHER_REGS>();
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
      // A: S^T(g) = K Q_g^T ; B: dP^T(g) = V dO_g^T  (M = 128 keys, N = 64, K = d) into buffer g % NB,
      // g counting query steps over all blocks
      auto issue_score = [&](uint32_t g) {
        const uint64_t so = static_cast<uint64_t>((g % NS) * C::Q_TILE) >> 4;
        const uint32_t tb = tmem + C::BUF(g % NB) + col;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint64_t oa = ((kk >> 2) * C::KV_CHUNK + (kk & 3) * 32) >> 4;
          const uint64_t ob = ((kk >> 2) * C::Q_CHUNK + (kk & 3) * 32) >> 4;
          mma_ss(tb, dKV_k + oa, dQO_k + so + ob, idesc_sdp, kk > 0 ? 1u : 0u);
        }
        mma_commit(b_sdp(g % NB));
      };
      // A: the buffer of step g still holds dQ^T(g - NB) until warps 8-11 have read it out
      auto score_ready = [&](uint32_t g) -> bool {
        if (!wait_bar(b_qfull(g % NS), (g / NS) & 1, p.timeout_ns, abort_flag, WB_QF)) return false;
        if (DQACC && role == 0 && g >= NB &&
            !wait_bar(b_dqfree(g % NB), ((g / NB) - 1) & 1, p.timeout_ns, abort_flag, WB_DQFREE))
          return false;
        return true;
      };
      int ix = blockIdx.x, iy = blockIdx.y;
      uint32_t gs = 0;  // query steps of the finished blocks
      int nb = 0;       // finished blocks
      bool ok = true;
      while (ok) {
        const Item w(ix, iy, p, D);
        if (!wait_bar(b_kv, nb & 1, p.timeout_ns, abort_flag, WB_KV)) break;
        if (role < 2) {
          if (!score_ready(gs)) break;
          tc_fence_after();
          issue_score(gs);
          for (int it = 0; ok && it < w.n_it; ++it) {
            const uint32_t g = gs + it, b = g % NB;
            if (it + 1 < w.n_it) {  // the next step's scores go to the other buffer first
              if (!score_ready(g + 1)) {
                ok = false;
                break;
              }
              tc_fence_after();
              issue_score(g + 1);
            }
            if (!wait_bar(b_ds(b), (g / NB) & 1, p.timeout_ns, abort_flag, WB_DS) ||
                (it == 0 && nb > 0 &&
                 !wait_bar(role == 0 ? b_vfree : b_kfree, (nb - 1) & 1, p.timeout_ns, abort_flag, WB_DONE))) {
              ok = false;
              break;
            }
            tc_fence_after();
            const int s = g % NS;
            const uint64_t so = static_cast<uint64_t>(s * C::Q_TILE) >> 4;
            const uint32_t tb = tmem + C::BUF(b) + col;
            const uint32_t acc0 = it > 0 ? 1u : 0u;
            // A: dV += P^T dO_g ; B: dK += dS^T Q_g  (M = 128 keys, N = d, K = 64; A from TMEM, B MN-major).
            // Packed P^T / dS^T of queries 16kk .. 16kk+15 sit at column (kk / 2) * 32 + (kk % 2) * 8.
#pragma unroll
            for (int kk = 0; kk < BQ / 16; ++kk)
              mma_ts(tmem + acc_col, tb + (kk >> 1) * 32 + (kk & 1) * 8, dOQ_mn + so + ((kk * 2048) >> 4),
                     idesc_acc, kk > 0 ? 1u : acc0);
            mma_commit(b_qempty(s));
            if (DQACC && role == 0) mma_commit(b_dvdone(b));
          }
        } else if constexpr (DQACC) {
          // C: dQ^T(g) = K^T dS^T(g) over S^T(g)'s columns (M = d, N = 64 queries, K = 128 keys)
          for (int it = 0; ok && it < w.n_it; ++it) {
            const uint32_t g = gs + it, b = g % NB;
            if (!wait_bar(b_ds(b), (g / NB) & 1, p.timeout_ns, abort_flag, WB_DS) ||
                !wait_bar(b_dvdone(b), (g / NB) & 1, p.timeout_ns, abort_flag, WB_DS)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t tb = tmem + C::BUF(b);
            const uint64_t bo = static_cast<uint64_t>(b * C::DS_TILE) >> 4;
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              mma_ss(tb, dK_mn + ((kk * 2048) >> 4), dDS_mn + bo + ((kk * 2048) >> 4), idesc_dq, kk > 0 ? 1u : 0u);
            mma_commit(b_dqfull(b));
          }
        }
        if (!ok) break;
        mma_commit(b_done);  // once these MMAs complete, dV / dK are final and K / V may be replaced
        gs += w.n_it;
        ok = next_item(nb++, true, ix, iy);
      }
      mma_commit(b_drain(role));
      wait_bar(b_drain(role), 0, p.timeout_ns, abort_flag, WB_DRAIN);
    }
    __syncwarp();
    tc_fence_before();
    __syncthreads();  // every role is done with TMEM
    if (warp == 13) {
      tc_fence_after();
      tmem_dealloc(tmem, 512);
    }
  } else if (warp < 8) {
    // ------------------------------------------------------------ elementwise: P^T, dS^T; dV epilogue
    setmaxnreg_inc<C::EW_REGS>();
    const int g = warp >> 2;          // column group: queries 32g .. 32g+31 of the tile
    const int k = threadIdx.x & 127;  // key within the tile == TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const float sl2 = p.scale_log2;
    int ix = blockIdx.x, iy = blockIdx.y;
    uint32_t gs = 0;
    int nb = 0;
    bool ok = true;
    while (ok) {
      const Item w(ix, iy, p, D);
      for (int it = 0; it < w.n_it; ++it) {
        const uint32_t gq = gs + it, b = gq % NB, s = gq % NS;
        if (!__all_sync(0xffffffffu, wait_bar(b_sdp(b), (gq / NB) & 1, p.timeout_ns, abort_flag, WB_SDP))) {
          ok = false;
          break;
        }
        // LSE/D of this stage were landed by the producer on q_full[s]; acquire them here too.
        if (!__all_sync(0xffffffffu, wait_bar(b_qfull(s), (gq / NS) & 1, p.timeout_ns, abort_flag, WB_QF))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t tS = tmem + lane_off + C::BUF(b), tDP = tS + 64;
        const float4* lse4 = reinterpret_cast<const float4*>(smem + C::OFF_LSE + s * BQ * 4) + 8 * g;
        const float4* dd4 = reinterpret_cast<const float4*>(smem + C::OFF_DD + s * BQ * 4) + 8 * g;
        int qh, qs;
        w.grp.step(it, w.it0, w.n_ith, qh, qs);
        const int q0 = qs * BQ + 32 * g;  // first query of this group's columns
        // masked: column c < kq (key > query, causal), q0 + c >= N (query past the sequence) or the
        // whole row when the key does not exist (past the sequence, or past the batch's key count:
        // a zero-filled K row gives S = 0, and exp(-LSE) need not be finite)
        const int klen = w.grp.klen;
        const bool need_mask = (CAUSAL && (q0 < w.key0 + 127)) || (q0 + 32 > N) || (w.key0 + 128 > klen);
        const int kq = CAUSAL ? (w.key0 + k - q0) : 0;
        const int qn = w.key0 + k < klen ? N - q0 : 0;
        uint32_t u[32], v[32];
        tmem_ld32_pair(tS + 32 * g, tDP + 32 * g, u, v);  // S^T and dP^T columns in one round trip
        float pv[32];
        // pairs of columns through the two-wide fp32 FMA / add / multiply (each lane rounds as the
        // scalar instruction would): fewer instructions in these issue-bound warps
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
        // Each group packs into the first half of its own 32 columns, never into columns the other
        // group may still be reading: queries 32g + 2c, 2c+1 go to column 32g + c.
        tmem_st16(tS + 32 * g, pk);
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
        tmem_st16(tDP + 32 * g, pk);
        if constexpr (DQACC) {
          // dS^T row k, queries 32g .. 32g+31: 16-byte units 4g .. 4g+3 of the 128-byte swizzled row
          uint8_t* row = smem + C::OFF_DS + b * C::DS_TILE + k * 128;
#pragma unroll
          for (int u4 = 0; u4 < 4; ++u4)
            *reinterpret_cast<uint4*>(row + (((4 * g + u4) ^ (k & 7)) << 4)) =
                make_uint4(pk[4 * u4], pk[4 * u4 + 1], pk[4 * u4 + 2], pk[4 * u4 + 3]);
          fence_proxy_async_smem();
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(b_ds(b));
      }
      if (!ok) break;
      gs += w.n_it;
      // ---------------------------------------------------------- dV epilogue: group g, columns g*D/2 ..
      if (!__all_sync(0xffffffffu, wait_bar(b_done, nb & 1, p.timeout_ns, abort_flag, WB_DONE))) break;
      tc_fence_after();
      {
        constexpr int HC = D / 2;  // columns per group
        uint32_t a[HC];
        if constexpr (HC == 64)
          tmem_ld64(tmem + lane_off + C::DV_COL + HC * g, a);
        else
          tmem_ld32(tmem + lane_off + C::DV_COL + HC * g, a);
        tc_fence_before();
        mbar_arrive(b_vfree);  // the next block's first dV MMA may overwrite the accumulator
        uint4* dst = reinterpret_cast<uint4*>(
            reinterpret_cast<uint16_t*>(p.dv) + (static_cast<size_t>(w.row_base) + w.key0 + k) * D + HC * g);
        const bool key_ok = w.key0 + k < N;  // keys past N exist only as zero rows of the block
#pragma unroll
        for (int u8 = 0; u8 < HC / 8; ++u8)
          if (key_ok) dst[u8] = make_uint4(bpack2<BF16>(__uint_as_float(a[8 * u8 + 0]), __uint_as_float(a[8 * u8 + 1])),
                               bpack2<BF16>(__uint_as_float(a[8 * u8 + 2]), __uint_as_float(a[8 * u8 + 3])),
                               bpack2<BF16>(__uint_as_float(a[8 * u8 + 4]), __uint_as_float(a[8 * u8 + 5])),
                               bpack2<BF16>(__uint_as_float(a[8 * u8 + 6]), __uint_as_float(a[8 * u8 + 7])));
      }
      int nx = -1, ny = 0;
      bool more = false;
      if ((threadIdx.x & 31) == 0) more = next_item(nb, true, nx, ny);
      more = __shfl_sync(0xffffffffu, more, 0);
      nx = __shfl_sync(0xffffffffu, nx, 0);
      ny = __shfl_sync(0xffffffffu, ny, 0);
      ++nb;
      if (!more) break;
      ix = nx;
      iy = ny;
    }
    tc_fence_before();
    __syncthreads();
  } else if (warp < 12) {
    // ------------------------------------------------------------ dQ read-out; dK epilogue
    // The four warps of this group meet at named barrier 2 once a step and at the dK epilogue, so
    // their control flow stays uniform: each of the group's barriers also ANDs every thread's "no
    // timeout" flag (bar.red.and), and thread 0 reads the item queue for the whole group.
    const int t = threadIdx.x - 256;  // TMEM lane = d index of dQ^T, key of dK
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    int ix = blockIdx.x, iy = blockIdx.y;
    uint32_t gs = 0;
    int nb = 0;
    bool ok = true;
    while (ok) {
      const Item w(ix, iy, p, D);
      for (int it = 0; DQACC && it < w.n_it; ++it) {
        const uint32_t gq = gs + it, b = gq % NB;
        const bool full =
            __all_sync(0xffffffffu, wait_bar(b_dqfull(b), (gq / NB) & 1, p.timeout_ns, abort_flag, WB_DQF));
        uint32_t u0[32], u1[32];
        if (full) {
          tc_fence_after();
          tmem_ld32_pair(tmem + lane_off + C::BUF(b), tmem + lane_off + C::BUF(b) + 32, u0, u1);
          tc_fence_before();
          mbar_arrive(b_dqfree(b));
        } else {
#pragma unroll
          for (int c = 0; c < 32; ++c) u0[c] = u1[c] = 0u;
        }
        if (!named_bar_and(2, 128, full && *abort_flag == 0u)) {
          ok = false;
          break;
        }
        if (t < D) {  // lanes >= d hold the zero-padded rows of dQ^T (d = 64)
          int qh, qs;
          w.grp.step(it, w.it0, w.n_ith, qh, qs);
          // lane t = d index, column c = query: a warp adds 32 consecutive floats of one query's row
          float* dst = p.dqacc + static_cast<size_t>(qh * p.Npad + qs * BQ) * D + t;
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            atomicAdd(dst + c * D, __uint_as_float(u0[c]));
            atomicAdd(dst + (32 + c) * D, __uint_as_float(u1[c]));
          }
        }
      }
      if (!ok) break;
      gs += w.n_it;
      // ---------------------------------------------------------- dK epilogue: dK = scale * accumulator
      const bool done = __all_sync(0xffffffffu, wait_bar(b_done, nb & 1, p.timeout_ns, abort_flag, WB_DONE));
      if (!named_bar_and(2, 128, done)) break;
      tc_fence_after();
      {
        uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<uint16_t*>(p.dk) +
                                              (static_cast<size_t>(w.row_base) + w.key0 + t) * D);
#pragma unroll 1
        for (int h = 0; h < D / 64; ++h) {
          uint32_t a[64];
          tmem_ld64(tmem + lane_off + C::DK_COL + 64 * h, a);
          if (h == D / 64 - 1) {
            tc_fence_before();
            mbar_arrive(b_kfree);  // the next block's first dK MMA may overwrite the accumulator
          }
          const float sc = p.scale;
          const bool key_ok = w.key0 + t < N;
#pragma unroll
          for (int u8 = 0; u8 < 8; ++u8)
            if (key_ok) dst[8 * h + u8] =
                make_uint4(bpack2<BF16>(__uint_as_float(a[8 * u8 + 0]) * sc, __uint_as_float(a[8 * u8 + 1]) * sc),
                           bpack2<BF16>(__uint_as_float(a[8 * u8 + 2]) * sc, __uint_as_float(a[8 * u8 + 3]) * sc),
                           bpack2<BF16>(__uint_as_float(a[8 * u8 + 4]) * sc, __uint_as_float(a[8 * u8 + 5]) * sc),
                           bpack2<BF16>(__uint_as_float(a[8 * u8 + 6]) * sc, __uint_as_float(a[8 * u8 + 7]) * sc));
        }
      }
      if (t == 0) {
        int nx = -1, ny = 0;
        const bool more = next_item(nb, true, nx, ny);
        dq_next[0] = more ? nx : -1;
        dq_next[1] = ny;
      }
      named_bar_sync(2, 128);
      ix = dq_next[0];
      iy = dq_next[1];
      ++nb;
      if (ix < 0) break;
      named_bar_sync(2, 128);  // every thread has read dq_next before thread 0 writes it again
    }
    tc_fence_before();
    __syncthreads();
  }
}

}  // namespace fa
