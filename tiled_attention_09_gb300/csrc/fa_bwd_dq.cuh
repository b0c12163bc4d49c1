// dQ as a separate pass of the backward (the alternative to accumulating dQ partials from the
// key-major main kernel), for d = 64 and 128.
//
// Method (page "transformer模型详解（十）：FlashAttention优化技术", section
// "Re-computation 而非缓存"): nothing of the N x N matrices is kept, so the pass
// rebuilds what dQ needs tile by tile, query-major: for a 128-row query tile i of one
// head and each 128-key tile j it may see,
//   S = Q_i K_j^T,  P = exp2(S * scale * log2 e - LSE_i * log2 e),
//   dP = dO_i V_j^T,  dS = P * (dP - D_i),  dQ_i += dS K_j,
// and finally dQ_i = scale * dQ_i. dQ stays in tensor memory for the whole row of
// tiles, so there is no fp32 accumulator in memory, no zeroing, no reductions and no
// conversion pass, and dQ is bitwise reproducible. The price is recomputing S and dP
// (two of the backward's five products) once more.
//
// Tensor memory: S_0, S_1 at 0 and 128 (a thread owns one query row, a TMEM lane; the
// packed 16-bit dS of a tile is written over the first half of each 64-key group of its
// S buffer and is the TMEM A operand of dQ += dS K), dP at 256, the dQ accumulator at
// 384 (d columns). Order of products per key tile j:
//   dP(j+1) once the elementwise warps have read dP(j); dQ(j) once they have written
//   dS(j); S(j+2) into S(j)'s buffer once dQ(j) has completed,
// so the tensor core works on tiles j+1 and j+2 while the elementwise warps turn tile j
// into dS. K tiles stream through a three-slot ring (a K tile is read by S(j) and, one
// tile later, by dQ(j)), V tiles through a one-slot ring (read by dP(j) only).
// Roles (12 warps): warps 0-7 elementwise (two groups of 64 key columns) and the dQ
// epilogue (each group half the head dimension), warp 8 TMA producer and work scheduler
// (cluster launch control takes over CTAs that have not started, as in the forward),
// warps 9, 10, 11 the MMA issuers of S, dP and dQ: one thread issues an MMA only every
// ~90-110 cycles, so a single issuer of the tile's 24 products would take about 2500
// cycles against 1536 of arithmetic.
#pragma once
#include "fa_bwd_main.cuh"

namespace fa {

template <int D_>
struct BwdDqCfg {
  static constexpr int D = D_, BQ = 128, BK = 128, NCH = D / 64;
  static constexpr int NSK = 3, NSV = (D == 64 ? 2 : 1);  // K and V ring slots
  static constexpr int CHUNK = 128 * 128;   // 128 rows x 64 elements
  static constexpr int TILE = 128 * D * 2;  // one 128-row tile
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_DO = OFF_Q + TILE;
  static constexpr int OFF_K = OFF_DO + TILE;
  static constexpr int OFF_V = OFF_K + NSK * TILE;
  static constexpr int OFF_LSE = OFF_V + NSV * TILE;  // 2 items x 128 floats
  static constexpr int OFF_DD = OFF_LSE + 2 * BQ * 4;  // 2 items x 128 floats
  static constexpr int OFF_BAR = OFF_DD + 2 * BQ * 4;
  // bars: q_full, q_free, kfull[NSK], kempty[NSK], vfull[NSV], vempty[NSV], s_full[2], ds_ready[2],
  // dq_done[2], dp_full, dp_free, dq_final, dq_read, clc, item_full[2], item_empty[2], drain[3]
  static constexpr int NBAR = 2 + 2 * NSK + 2 * NSV + 6 + 4 + 1 + 4 + 3;
  static constexpr int BAR_BYTES = (NBAR * 8 + 15) & ~15;
  static constexpr int SMEM_BYTES = 1024 + OFF_BAR + BAR_BYTES + 16 + 16 + 16;
  static constexpr int THREADS = 384;
  static constexpr uint32_t S_COL0 = 0, DP_COL = 256, DQ_COL = 384;
  static_assert(D == 64 || D == 128, "d = 64 or 128");
  static_assert(SMEM_BYTES <= 232448, "smem budget");
};

// where-codes of this kernel's waits (60-69)
enum : uint32_t { WQ_Q = 60, WQ_KV = 61, WQ_S = 62, WQ_DS = 63, WQ_DP = 64, WQ_DQ = 65, WQ_ITEM = 66, WQ_CLC = 67,
                  WQ_DRAIN = 68 };

// One work item: the 128-row query tile y of query head x (blockIdx of the CTA launched for it; under
// causal masking y = 0 is the last, longest tile, so the launch order is longest-first).
template <bool CAUSAL, bool GRP>
struct BwdDqItem {
  int qh;      // query head (b, h): the z coordinate of the Q and dO maps
  int kvh;     // its K/V head (b, h / G)
  int q0;      // first query row of the tile within the head
  int klen;    // keys that exist for this batch: min(N, kv_len[b]), or N
  int ntile;   // key tiles the tile sees (0: a tile whose queries see no key gets dQ = 0)
  __device__ __forceinline__ BwdDqItem(int x, int y, const BwdParams& p) {
    const int n_qt = (p.N + 127) / 128;
    const int qt = CAUSAL ? n_qt - 1 - y : y;
    qh = x;
    q0 = qt * 128;
    if constexpr (GRP) {
      const int G = p.H / p.Hkv;
      const int b = x / p.H;
      kvh = b * p.Hkv + (x - b * p.H) / G;
      klen = bwd_key_count(p, b);
    } else {
      kvh = x;
      klen = p.N;
    }
    const int nk = (klen + 127) / 128;
    ntile = CAUSAL ? (qt + 1 < nk ? qt + 1 : nk) : nk;
  }
};

template <int D_, bool BF16, bool CAUSAL, bool GRP>
__global__ void __launch_bounds__(384, 1) fa_bwd_dq_kernel(const __grid_constant__ BwdParams p) {
  using C = BwdDqCfg<D_>;
  using Item = BwdDqItem<CAUSAL, GRP>;
  constexpr int D = C::D, NSK = C::NSK, NSV = C::NSV;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t s0 = smem_u32(smem);
  const uint32_t sQ = s0 + C::OFF_Q, sDO = s0 + C::OFF_DO, sK = s0 + C::OFF_K, sV = s0 + C::OFF_V;
  uint8_t* aux = smem + C::OFF_BAR;
  uint64_t* bars = reinterpret_cast<uint64_t*>(aux);
  const uint32_t b_qfull = smem_u32(&bars[0]);
  const uint32_t b_qfree = smem_u32(&bars[1]);
  auto b_kfull = [&](int s) { return smem_u32(&bars[2 + s]); };
  auto b_kempty = [&](int s) { return smem_u32(&bars[2 + NSK + s]); };
  auto b_vfull = [&](int s) { return smem_u32(&bars[2 + 2 * NSK + s]); };
  auto b_vempty = [&](int s) { return smem_u32(&bars[2 + 2 * NSK + NSV + s]); };
  constexpr int B0 = 2 + 2 * NSK + 2 * NSV;
  auto b_sfull = [&](int b) { return smem_u32(&bars[B0 + b]); };
  auto b_dsready = [&](int b) { return smem_u32(&bars[B0 + 2 + b]); };
  auto b_dqdone = [&](int b) { return smem_u32(&bars[B0 + 4 + b]); };
  const uint32_t b_dpfull = smem_u32(&bars[B0 + 6]);
  const uint32_t b_dpfree = smem_u32(&bars[B0 + 7]);
  const uint32_t b_dqfinal = smem_u32(&bars[B0 + 8]);
  const uint32_t b_dqread = smem_u32(&bars[B0 + 9]);
  const uint32_t b_clc = smem_u32(&bars[B0 + 10]);
  auto b_item_full = [&](int i) { return smem_u32(&bars[B0 + 11 + i]); };
  auto b_item_empty = [&](int i) { return smem_u32(&bars[B0 + 13 + i]); };
  auto b_drain = [&](int i) { return smem_u32(&bars[B0 + 15 + i]); };
  const uint32_t clc_resp = smem_u32(aux + C::BAR_BYTES);
  volatile int* items = reinterpret_cast<volatile int*>(aux + C::BAR_BYTES + 16);  // [2][2]: x, y (x < 0: none)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(aux + C::BAR_BYTES + 32);
  volatile uint32_t* abort_flag = tmem_slot + 1;

  const int warp = threadIdx.x >> 5;
  const int N = p.N;

  if (threadIdx.x == 0) {
    mbar_init(b_qfull, 1);
    // the S issuer after its item's last S, the dP issuer after its last dP, and each elementwise warp
    // once it has taken the item's Q stage: without these eight, issuers two short items ahead of the
    // elementwise warps would let q_full complete twice past a parity those warps still wait for
    mbar_init(b_qfree, 2 + 8);
    for (int s = 0; s < NSK; ++s) {
      mbar_init(b_kfull(s), 1);
      mbar_init(b_kempty(s), 1);
    }
    for (int s = 0; s < NSV; ++s) {
      mbar_init(b_vfull(s), 1);
      mbar_init(b_vempty(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(b_sfull(b), 1);
      mbar_init(b_dsready(b), 8);  // one arrival per elementwise warp
      mbar_init(b_dqdone(b), 1);
    }
    mbar_init(b_dpfull, 1);
    mbar_init(b_dpfree, 8);
    mbar_init(b_dqfinal, 1);
    mbar_init(b_dqread, 8);
    mbar_init(b_clc, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(b_item_full(i), 1);
      mbar_init(b_item_empty(i), 3 + 8);  // the three MMA threads and one lane per elementwise warp
    }
    for (int i = 0; i < 3; ++i) mbar_init(b_drain(i), 1);
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

  // Work loop shared by all roles: the CTA starts with the tile it was launched for; the producer
  // takes over not-yet-launched CTAs (cluster launch control, asked with the item's last K/V
  // loads) and passes their ids through a two-entry queue; an id x < 0 ends the loop. Barrier
  // phases run on per-role counters across items.
  if (warp == 8) {
    // ------------------------------------------------------------ producer
    if (elect_one()) {
      tma_prefetch_desc(&p.tm_q);
      tma_prefetch_desc(&p.tm_do);
      tma_prefetch_desc(&p.tm_k);
      tma_prefetch_desc(&p.tm_v);
      int ix = blockIdx.x, iy = blockIdx.y;
      uint32_t nkl = 0, nvl = 0;  // K and V tiles issued (ring positions)
      int n_items = 0;
      bool clc_live = true, clc_pending = false, ok = true;
      uint32_t clc_phase = 0;
      auto ask = [&]() {
        if (!clc_live) return;
        fence_proxy_async_smem();  // earlier generic reads of the answer slot come first
        mbar_arrive_expect_tx(b_clc, 16);
        clc_try_cancel(clc_resp, b_clc);
        clc_pending = true;
      };
      while (ok) {
        const Item w(ix, iy, p);
        // Q, dO of the previous item are dead once its last S and dP products have completed and every
        // elementwise warp has taken its stage (and LSE / D buffer)
        if (n_items > 0 && !wait_bar(b_qfree, (n_items - 1) & 1, p.timeout_ns, abort_flag, WQ_Q)) break;
        const int li = n_items & 1;  // LSE / D buffer of this item
        const int qrow = w.qh * p.Npad + w.q0;
        mbar_arrive_expect_tx(b_qfull, 2 * C::TILE + 2 * C::BQ * 4);
#pragma unroll
        for (int c = 0; c < C::NCH; ++c)
#pragma unroll
          for (int r = 0; r < 2; ++r) {  // the 64-row boxes of the query maps
            tma_load_3d(sQ + c * C::CHUNK + r * 8192, &p.tm_q, b_qfull, c * 64, w.q0 + 64 * r, w.qh);
            tma_load_3d(sDO + c * C::CHUNK + r * 8192, &p.tm_do, b_qfull, c * 64, w.q0 + 64 * r, w.qh);
          }
        bulk_load(s0 + C::OFF_LSE + li * C::BQ * 4, p.lse2 + qrow, C::BQ * 4, b_qfull);
        bulk_load(s0 + C::OFF_DD + li * C::BQ * 4, p.Dvec + qrow, C::BQ * 4, b_qfull);
        ++n_items;
        if (w.ntile == 0) ask();
        for (int j = 0; j < w.ntile; ++j) {
          if (j == w.ntile - 1) ask();
          {
            const uint32_t s = nkl % NSK, use = nkl / NSK;
            if (use > 0 && !wait_bar(b_kempty(s), (use - 1) & 1, p.timeout_ns, abort_flag, WQ_KV)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(b_kfull(s), C::TILE);
#pragma unroll
            for (int c = 0; c < C::NCH; ++c)
              tma_load_3d(sK + s * C::TILE + c * C::CHUNK, &p.tm_k, b_kfull(s), c * 64, j * 128, w.kvh);
            ++nkl;
          }
          {
            const uint32_t s = nvl % NSV, use = nvl / NSV;
            if (use > 0 && !wait_bar(b_vempty(s), (use - 1) & 1, p.timeout_ns, abort_flag, WQ_KV)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(b_vfull(s), C::TILE);
#pragma unroll
            for (int c = 0; c < C::NCH; ++c)
              tma_load_3d(sV + s * C::TILE + c * C::CHUNK, &p.tm_v, b_vfull(s), c * 64, j * 128, w.kvh);
            ++nvl;
          }
        }
        if (!ok) break;
        int nx = -1, ny = 0;
        if (clc_live) {
          if (!wait_bar(b_clc, clc_phase, p.timeout_ns, abort_flag, WQ_CLC)) break;
          clc_pending = false;
          clc_phase ^= 1u;
          if (!clc_query(clc_resp, nx, ny)) {
            clc_live = false;
            nx = -1;
          } else if (nx < 0 || ny < 0 || nx >= static_cast<int>(gridDim.x) || ny >= static_cast<int>(gridDim.y)) {
            report_status(FA_DEV_BAD_INDEX, WQ_CLC);  // a taken-over CTA must be one of this grid's
            clc_live = false;
            nx = -1;
          }
        }
        const int qi = n_items - 1;  // queue entry qi names the item after item qi
        if (qi >= 2 && !wait_bar(b_item_empty(qi & 1), ((qi >> 1) - 1) & 1, p.timeout_ns, abort_flag, WQ_ITEM))
          break;
        items[2 * (qi & 1)] = nx;
        items[2 * (qi & 1) + 1] = ny;
        mbar_arrive(b_item_full(qi & 1));  // release: readers acquire through their wait
        if (nx < 0) break;
        ix = nx;
        iy = ny;
      }
      // Drain: every issued copy has landed before the CTA may exit.
      if (clc_pending) wait_bar(b_clc, clc_phase, p.timeout_ns, abort_flag, WQ_DRAIN);
      if (n_items > 0) wait_bar(b_qfull, (n_items - 1) & 1, p.timeout_ns, abort_flag, WQ_DRAIN);
      for (uint32_t u = (nkl > NSK ? nkl - NSK : 0u); u < nkl; ++u)
        wait_bar(b_kfull(u % NSK), (u / NSK) & 1, p.timeout_ns, abort_flag, WQ_DRAIN);
      for (uint32_t u = (nvl > NSV ? nvl - NSV : 0u); u < nvl; ++u)
        wait_bar(b_vfull(u % NSV), (u / NSV) & 1, p.timeout_ns, abort_flag, WQ_DRAIN);
    }
    __syncwarp();
    tc_fence_before();
    __syncthreads();
  } else if (warp >= 9) {
    // ------------------------------------------------------------ MMA issuers: 9 = S, 10 = dP, 11 = dQ
    const int role = warp - 9;
    if (elect_one()) {
      constexpr uint32_t idesc_s = make_idesc(128, 128, BF16, false, false);
      constexpr uint32_t idesc_dq = make_idesc(128, D, BF16, false, true);
      // Descriptors are built once; an MMA only adds (byte offset >> 4) to the start-address field.
      const uint64_t dq_k = make_sdesc(sQ, 16, 1024);          // Q, K-major (rows = queries)
      const uint64_t ddo_k = make_sdesc(sDO, 16, 1024);        // dO, K-major
      const uint64_t dk_k = make_sdesc(sK, 16, 1024);          // K in a ring slot, K-major (rows = keys)
      const uint64_t dv_k = make_sdesc(sV, 16, 1024);          // V in a ring slot, K-major
      const uint64_t dk_mn = make_sdesc(sK, C::CHUNK, 1024);   // K as the MN-major B of dS K (N = d)
      int ix = blockIdx.x, iy = blockIdx.y;
      uint32_t kseq = 0, vseq = 0;  // ring positions of the item's first K and V tiles
      uint32_t ns = 0;              // S products issued (all items): S buffer ns & 1
      uint32_t ndp = 0;             // dP products issued
      uint32_t ndq = 0;             // dQ products issued (= dS tiles consumed)
      int n_items = 0;
      bool ok = true;
      // S(j) = Q K_j^T into S buffer (ns & 1); dP(j) = dO V_j^T (M = 128 queries, N = 128 keys, K = d)
      auto issue_s = [&](int j) -> bool {
        const uint32_t b = ns & 1, ks = (kseq + j) % NSK, ku = (kseq + j) / NSK;
        if (!wait_bar(b_kfull(ks), ku & 1, p.timeout_ns, abort_flag, WQ_KV)) return false;
        // the buffer held dS of two products ago: its dQ must have completed
        if (ns >= 2 && !wait_bar(b_dqdone(b), ((ns >> 1) - 1) & 1, p.timeout_ns, abort_flag, WQ_DQ)) return false;
        tc_fence_after();
        const uint64_t ko = static_cast<uint64_t>(ks * C::TILE) >> 4;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint64_t off = static_cast<uint64_t>(((kk >> 2) * C::CHUNK + (kk & 3) * 32) >> 4);
          mma_ss(tmem + C::S_COL0 + 128 * b, dq_k + off, dk_k + ko + off, idesc_s, kk > 0 ? 1u : 0u);
        }
        mma_commit(b_sfull(b));
        ++ns;
        return true;
      };
      auto issue_dp = [&](int j) -> bool {
        const uint32_t vs = (vseq + j) % NSV, vu = (vseq + j) / NSV;
        if (!wait_bar(b_vfull(vs), vu & 1, p.timeout_ns, abort_flag, WQ_KV)) return false;
        // the elementwise warps have read the previous dP
        if (ndp > 0 && !wait_bar(b_dpfree, (ndp - 1) & 1, p.timeout_ns, abort_flag, WQ_DP)) return false;
        tc_fence_after();
        const uint64_t vo = static_cast<uint64_t>(vs * C::TILE) >> 4;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint64_t off = static_cast<uint64_t>(((kk >> 2) * C::CHUNK + (kk & 3) * 32) >> 4);
          mma_ss(tmem + C::DP_COL, ddo_k + off, dv_k + vo + off, idesc_s, kk > 0 ? 1u : 0u);
        }
        mma_commit(b_dpfull);
        mma_commit(b_vempty(vs));
        ++ndp;
        return true;
      };
      // dQ += dS(j) K_j: A = packed dS from the S buffer (keys 16kk.. at column 64 (kk / 4) + 8 (kk % 4)),
      // B = K_j MN-major (M = 128 queries, N = d, K = 128 keys)
      auto issue_dq = [&](int j, bool first) -> bool {
        const uint32_t b = ndq & 1, ks = (kseq + j) % NSK, ku = (kseq + j) / NSK;
        if (!wait_bar(b_dsready(b), (ndq >> 1) & 1, p.timeout_ns, abort_flag, WQ_DS)) return false;
        // K_j landed long before (S(j) read it); this thread acquires the copy for its own products
        if (!wait_bar(b_kfull(ks), ku & 1, p.timeout_ns, abort_flag, WQ_KV)) return false;
        // the first product of an item overwrites the accumulator: the previous epilogue has read it
        if (first && n_items > 0 && !wait_bar(b_dqread, (n_items - 1) & 1, p.timeout_ns, abort_flag, WQ_DQ))
          return false;
        tc_fence_after();
        const uint64_t ko = static_cast<uint64_t>(ks * C::TILE) >> 4;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_ts(tmem + C::DQ_COL, tmem + C::S_COL0 + 128 * b + (kk >> 2) * 64 + (kk & 3) * 8,
                 dk_mn + ko + static_cast<uint64_t>((kk * 2048) >> 4), idesc_dq, (first && kk == 0) ? 0u : 1u);
        mma_commit(b_dqdone(b));
        mma_commit(b_kempty(ks));
        ++ndq;
        return true;
      };
      // S(j) waits for its K tile and, from the third tile on, for dQ(j - 2) (its buffer held dS(j - 2));
      // dP(j) for its V tile and for the elementwise warps to have read dP(j - 1); dQ(j) for dS(j).
      while (ok) {
        const Item w(ix, iy, p);
        const int nt = w.ntile;
        if (role < 2 && !wait_bar(b_qfull, n_items & 1, p.timeout_ns, abort_flag, WQ_Q)) break;
        for (int j = 0; ok && j < nt; ++j) {
          if (role == 0)
            ok = issue_s(j);
          else if (role == 1)
            ok = issue_dp(j);
          else
            ok = issue_dq(j, j == 0);
        }
        if (!ok) break;
        if (role < 2) mma_commit(b_qfree);  // every S (dP) of the item has been issued
        if (role == 2) mma_commit(b_dqfinal);  // the item's dQ is complete (no key tile: nothing to wait for)
        kseq += nt;
        vseq += nt;
        const int qi = n_items++;
        if (!wait_bar(b_item_full(qi & 1), (qi >> 1) & 1, p.timeout_ns, abort_flag, WQ_ITEM)) break;
        const int nx = items[2 * (qi & 1)], ny = items[2 * (qi & 1) + 1];
        mbar_arrive(b_item_empty(qi & 1));
        if (nx < 0) break;
        ix = nx;
        iy = ny;
      }
      // Drain: all issued MMAs complete before teardown.
      mma_commit(b_drain(role));
      wait_bar(b_drain(role), 0, p.timeout_ns, abort_flag, WQ_DRAIN);
    }
    __syncwarp();
    tc_fence_before();
    __syncthreads();  // every role is done with TMEM
    if (warp == 9) {
      tc_fence_after();
      tmem_dealloc(tmem, 512);
    }
  } else if (warp < 8) {
    // ------------------------------------------------------------ elementwise: dS; dQ epilogue
    const int grp = warp >> 2;        // key columns 64 grp .. 64 grp + 63 of each tile
    const int r = threadIdx.x & 127;  // query row within the tile == TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const bool lane0 = (threadIdx.x & 31) == 0;
    const float sl2 = p.scale_log2;
    int ix = blockIdx.x, iy = blockIdx.y;
    uint32_t nt_all = 0;  // tiles consumed (all items): S buffer nt_all & 1
    int n_items = 0;
    bool ok = true;
    while (ok) {
      const Item w(ix, iy, p);
      const int li = n_items & 1;
      if (!__all_sync(0xffffffffu, wait_bar(b_qfull, n_items & 1, p.timeout_ns, abort_flag, WQ_Q))) break;
      const float lse2 = reinterpret_cast<const float*>(smem + C::OFF_LSE + li * C::BQ * 4)[r];
      const float dd = reinterpret_cast<const float*>(smem + C::OFF_DD + li * C::BQ * 4)[r];
      __syncwarp();
      if (lane0) mbar_arrive(b_qfree);  // this warp has passed q_full of the item (and read LSE, D)
      const int q = w.q0 + r;  // query row within the head
      // keys this row may see: those that exist, and (causal) none past the query itself
      const int klim = (CAUSAL && w.klen > q + 1) ? q + 1 : w.klen;
      for (int j = 0; j < w.ntile; ++j, ++nt_all) {
        const uint32_t b = nt_all & 1;
        if (!__all_sync(0xffffffffu, wait_bar(b_sfull(b), (nt_all >> 1) & 1, p.timeout_ns, abort_flag, WQ_S)) ||
            !__all_sync(0xffffffffu, wait_bar(b_dpfull, nt_all & 1, p.timeout_ns, abort_flag, WQ_DP))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t tS = tmem + lane_off + C::S_COL0 + 128 * b + 64 * grp;
        const uint32_t tDP = tmem + lane_off + C::DP_COL + 64 * grp;
        // keys of this group past klim (causal diagonal, past the sequence, key padding) are masked
        const int lim = klim - (j * 128 + 64 * grp);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t sv[32], dv[32];
          tmem_ld32_pair(tS + 32 * h, tDP + 32 * h, sv, dv);
          if (h == 1) {
            tc_fence_before();
            __syncwarp();
            if (lane0) mbar_arrive(b_dpfree);  // dP(j + 1) may overwrite the columns
          }
          uint32_t pk[16];
#pragma unroll
          for (int c = 0; c < 16; ++c) {
            const int k0 = 32 * h + 2 * c;
            float x0 = ex2_approx(fmaf(__uint_as_float(sv[2 * c]), sl2, -lse2));
            float x1 = ex2_approx(fmaf(__uint_as_float(sv[2 * c + 1]), sl2, -lse2));
            x0 = k0 < lim ? x0 : 0.f;
            x1 = k0 + 1 < lim ? x1 : 0.f;
            pk[c] = bpack2<BF16>(x0 * (__uint_as_float(dv[2 * c]) - dd), x1 * (__uint_as_float(dv[2 * c + 1]) - dd));
          }
          // keys 64 grp + 2c, 2c+1 go to column 64 grp + c of the S buffer: half h writes columns
          // 16h .. 16h + 15 of the group, which its first half has already read
          tmem_st16(tS + 16 * h, pk);
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane0) mbar_arrive(b_dsready(b));
      }
      if (!ok) break;
      // ---------------------------------------------------------- dQ epilogue: group grp, columns grp*D/2 ..
      if (!__all_sync(0xffffffffu, wait_bar(b_dqfinal, n_items & 1, p.timeout_ns, abort_flag, WQ_DQ))) break;
      tc_fence_after();
      {
        constexpr int HC = D / 2;  // columns per group
        uint32_t a[HC];
        if (w.ntile > 0) {
          if constexpr (HC == 64)
            tmem_ld64(tmem + lane_off + C::DQ_COL + HC * grp, a);
          else
            tmem_ld32(tmem + lane_off + C::DQ_COL + HC * grp, a);
        } else {
#pragma unroll
          for (int c = 0; c < HC; ++c) a[c] = 0u;  // no key: dQ = 0 (the accumulator was never written)
        }
        tc_fence_before();
        __syncwarp();
        if (lane0) mbar_arrive(b_dqread);  // the next item's first dQ product may overwrite the accumulator
        const float sc = p.scale;
        if (q < N) {
          uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<uint16_t*>(p.dq) +
                                                (static_cast<size_t>(w.qh) * N + q) * D + HC * grp);
#pragma unroll
          for (int u8 = 0; u8 < HC / 8; ++u8)
            dst[u8] = make_uint4(bpack2<BF16>(__uint_as_float(a[8 * u8 + 0]) * sc, __uint_as_float(a[8 * u8 + 1]) * sc),
                                 bpack2<BF16>(__uint_as_float(a[8 * u8 + 2]) * sc, __uint_as_float(a[8 * u8 + 3]) * sc),
                                 bpack2<BF16>(__uint_as_float(a[8 * u8 + 4]) * sc, __uint_as_float(a[8 * u8 + 5]) * sc),
                                 bpack2<BF16>(__uint_as_float(a[8 * u8 + 6]) * sc, __uint_as_float(a[8 * u8 + 7]) * sc));
        }
      }
      const int qi = n_items++;
      if (!__all_sync(0xffffffffu, wait_bar(b_item_full(qi & 1), (qi >> 1) & 1, p.timeout_ns, abort_flag, WQ_ITEM)))
        break;
      const int nx = items[2 * (qi & 1)], ny = items[2 * (qi & 1) + 1];
      __syncwarp();
      if (lane0) mbar_arrive(b_item_empty(qi & 1));
      if (nx < 0) break;
      ix = nx;
      iy = ny;
    }
    tc_fence_before();
    __syncthreads();
  }
}

}  // namespace fa
