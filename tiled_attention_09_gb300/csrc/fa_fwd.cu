// Fused attention forward for sm_103a (K1).
//
// Method (page "transformer模型详解（十）：FlashAttention优化技术"): one kernel keeps
// every intermediate on chip ("Kernel Fusion"), walks the scores in B_q x B_k
// tiles ("Tiling 分块策略") and runs the online softmax of that section: per
// tile the local row max and exponential sum, an update of the running max
// with a rescale of the running sum and of the output accumulator, and one
// normalisation at the end. Only O and the per-row log-sum-exp go to HBM.
//
// GB300 design. A work item is NT query tiles of 128 rows of one (b, h) head
// (NT = 2 for d <= 128, 1 for d = 256; with short rows or few heads the host may
// run d <= 128 with one tile an item, FwdParams::tpi); the item streams the head's K/V tiles
// of 128 keys through a ring of shared-memory slots filled by TMA. The kernel
// is persistent in the Blackwell way: the grid has one CTA per item, but a
// running CTA takes over CTAs that have not been launched yet (cluster launch
// control) instead of exiting, so Q/K loads, TMEM allocation and the first
// S = Q K^T of the next item overlap the end of the current one, and the
// hardware's launch order (heaviest query blocks first under causal masking)
// is kept. Roles:
//   warps 0..4NT-1  softmax + epilogue: one warpgroup per query tile; thread r
//                   owns row r of S, P and O in tensor memory (TMEM lane r), so
//                   row max and row sum need no shuffles.
//   warp 4NT        producer: TMA loads of Q_t and K_j, V_j (ring order
//                   K0 V0 K1 V1 ...); asks for the next item and passes its id
//                   to the other roles through a two-entry queue.
//   warp 4NT+1      MMA issuer: tcgen05.mma S_t = Q_t K_j^T (both operands in
//                   smem) and O_t += P_t V_j (P from TMEM, V from smem), with
//                   tcgen05.commit arrivals on mbarriers.
//   warps 4NT+2..   idle (they complete the last warpgroup).
// With NT = 2 the block is launched with 168 registers a thread (three warps
// per SM sub-partition) and setmaxnreg moves them to the softmax warpgroups
// (216) from the producer/MMA warpgroup (72).
// TMEM columns: S_t at 128t (fp32 128x128; P_t as 16-bit pairs over its first
// 64 columns), O_t at 256 + d*t (fp32 128 x d).
// Issue order per key tile j: PV_0(j-1), S_0(j), PV_1(j-1), S_1(j); the commit
// that announces S_t(j) also covers PV_t(j-1), so when the softmax sees S_t(j)
// the accumulator O_t is quiescent and can be rescaled in place.
// Rescaling is lazy: the running max m used for the exponentials only moves when
// the row max grows by more than 2^8. From the second key tile on, the softmax
// exponentiates against the current m and finds the new row max in the same
// pass; only a row whose max grew past the threshold rescales O and repeats the
// pass. The final O / l and LSE use the same m, so the result is exact up to
// rounding. With a lazy max, the largest probability of a key tile is 2^delta
// (0 < delta <= 8) rather than exactly 1, and its rounding to the dtype for the
// P V product would not cancel in acc / l: for a nearly one-hot row that is an
// error of up to half an ulp of P times |V|. So O is divided by l plus the
// rounding error of each tile's largest probability (one exponential per row
// and tile), which gives a one-hot row its V row again; the LSE keeps l.
// Causal: tiles above the diagonal are never loaded or computed; the
// diagonal tile masks keys > query inside the softmax.
#include <cuda.h>
#include <type_traits>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "common.cuh"
#include "fa_bwd_order.cuh"
#include "launch.h"

namespace fa {
namespace {

struct FwdParams {
  CUtensorMap tm_q, tm_k, tm_v;  // Q over B*H heads; K, V over B*Hkv heads
  uint16_t* o;     // [B*H*N, d] in the input dtype (nullptr when o32 is given)
  float* o32;      // optional [B*H*N, d] fp32 output instead of o
  float* lse;      // [B*H*N]
  uint16_t* o_lo;  // optional [B*H*N, d]: dtype(O_fp32 - float(O)), the rounding residual of O
  const int* kv_len;  // optional [B]: batch b attends only to keys j < kv_len[b] (key padding)
  float* part_o;      // split keys (kv_splits > 1): [kv_splits][B*H*N, d] fp32 partial O, each normalised
  float* part_lse;    // [kv_splits][B*H*N] natural-log LSE of each part (-inf: the part saw no key)
  long long part_rows;  // B*H*N
  int kv_splits;      // CTAs that share one query block's key range (1: no split)
  int tpi;            // query tiles per work item: NT, or 1 (short rows: twice the items, each half as long)
  int N;
  int H, G;        // query heads; query heads per K/V head
  int n_qblk;
  float scale_log2;
  float rescale_threshold;
  unsigned long long timeout_ns;
};

template <int D>
struct FwdCfg {
  static constexpr int NT = (D <= 128) ? 2 : 1;                   // query tiles per work item
  static constexpr int CHUNK = 128 * 128;                         // 128 rows x 64 elems x 2 B
  static constexpr int NCHUNK = D / 64;
  static constexpr int TILE = 128 * D * 2;                        // one 128-row tile
  static constexpr int NS = (D == 64) ? 6 : (D == 128 ? 4 : 2);   // ring slots
  static constexpr int SMEM_Q = NT * TILE;
  // d = 64 and 256: P_t gets its own TMEM columns (d = 64: O_t is only 64 wide; d = 256: one query
  // tile leaves 128 columns between S and O), and S_t(j+1) can be computed as soon as the softmax has
  // read S_t(j), while P_t(j) is still being formed
  static constexpr bool SEP_P = D == 64 || D == 256;
  static constexpr int SMEM_RING = NS * TILE;
  // q, qfree, full[NS], empty[NS], s[NT], p[NT], o[NT], ofree[NT], clc, item_full[2], item_empty[2], drain,
  // and with SEP_P sfree[NT], pv[NT]
  static constexpr int NBAR = 2 + 2 * NS + 4 * NT + 1 + 4 + 1 + (SEP_P ? 2 * NT : 0);
  static constexpr int BAR_BYTES = (NBAR * 8 + 15) & ~15;
  // after the barriers: the 16-byte launch-control answer, the item queue (2 x {x, y}), TMEM slot + abort flag
  static constexpr int SMEM_BYTES = 1024 + SMEM_Q + SMEM_RING + BAR_BYTES + 16 + 16 + 16;
  // NT softmax warpgroups + one warpgroup with the producer, the MMA issuer and two idle warps
  static constexpr int THREADS = 128 * NT + 128;
  // Register split (NT = 2): launched with LAUNCH_REGS per thread (three warps per SM
  // sub-partition), the softmax warpgroups then take SOFTMAX_REGS and the other
  // warpgroup keeps OTHER_REGS. The host refuses to launch unless the compiled
  // count equals LAUNCH_REGS, so the increase always finds its registers.
  static constexpr int LAUNCH_REGS = 168;
  static constexpr int SOFTMAX_REGS = 216;
  static constexpr int OTHER_REGS = 72;
  static_assert(NT == 1 || 128 * NT * SOFTMAX_REGS + 128 * OTHER_REGS <= THREADS * LAUNCH_REGS, "register split");
  static constexpr uint32_t TMEM_COLS = 512;
  __host__ __device__ static constexpr uint32_t S_COL(int t) { return 128u * t; }
  __host__ __device__ static constexpr uint32_t O_COL(int t) { return 256u + D * t; }
  // packed 16-bit P_t: over S_t's first 64 columns, or (SEP_P) in its own 64 columns: after O (d = 64),
  // between S and O (d = 256)
  __host__ __device__ static constexpr uint32_t P_COL(int t) {
    return SEP_P ? (D == 64 ? 256u + NT * D + 64u * t : 128u + 64u * t) : S_COL(t);
  }
  static_assert(!SEP_P || D == 64 || P_COL(NT - 1) + 64 <= O_COL(0), "P between S and O");
  static_assert(O_COL(NT - 1) + D <= TMEM_COLS, "TMEM budget");
  static_assert(P_COL(NT - 1) + 64 <= TMEM_COLS, "TMEM budget");
  static_assert(SMEM_BYTES <= 227 * 1024, "smem budget");
};

// One work item: p.tpi (NT, or 1) consecutive query tiles of one (b, h) head, named by the
// blockIdx of the CTA that was launched for it (x = head, y = launch rank x key
// split; under causal masking rank 0 is the last and heaviest query block, so the
// hardware's launch order is longest-first; for d = 256 without a split the kernel
// maps the launch index through the backward's order first, see item_order). With split keys (kv_splits = S > 1)
// the item is one of S contiguous ranges of the block's key tiles, [kt0, kt1):
// each range writes its own normalised partial O and LSE and a merge pass joins
// them by the online-softmax rule (O = sum_s e^(LSE_s - LSE) O_s).
template <int NT, bool CAUSAL, bool SPLIT>
struct FwdItem {
  int bh;        // query head (b, h): the z coordinate of the Q map
  int bkv;       // its K/V head (b, h / G): the z coordinate of the K and V maps
  int q_row0;    // first query row of the item within the head
  int row_base;  // row of (b, h, 0) in the [B*H*N, d] view
  int klen;      // keys that exist for this batch: min(N, kv_len[b]), or N
  int nk;        // key tiles that hold them (at least one: a row with no key gets O = 0, LSE = -inf)
  int n_valid;   // query tiles that exist (the last block can hold one tile fewer)
  int nmax;      // key tiles streamed for the item
  int n_t[NT];   // key tiles that tile t needs
  int kt0, kt1;  // the item's range of key tiles (all of them without a split)
  int sp;        // which of the kv_splits ranges (0 without a split)
  __device__ __forceinline__ FwdItem(int x, int y, const FwdParams& p) {
    const int N = p.N;
    const int S = SPLIT ? p.kv_splits : 1;
    const int rank = SPLIT ? y / S : y;
    sp = SPLIT ? y - rank * S : 0;
    const int qb = CAUSAL ? (p.n_qblk - 1 - rank) : rank;
    bh = x;
    const int b = x / p.H;
    bkv = b * (p.H / p.G) + (x - b * p.H) / p.G;
    klen = N;
    if (p.kv_len) {
      const int l = __ldg(p.kv_len + b);
      klen = l < 0 ? 0 : (l > N ? N : l);
    }
    nk = klen > 0 ? (klen + 127) / 128 : 1;
    q_row0 = qb * 128 * p.tpi;
    row_base = x * N;
    n_valid = (N - q_row0 + 127) / 128;  // a tile that runs past N still exists (its tail is masked)
    if (n_valid > p.tpi) n_valid = p.tpi;  // with one tile an item, tile 1's warpgroup sits the item out
    kt0 = 0;
    kt1 = 1 << 30;
    if constexpr (SPLIT) {
      int full = 0;
#pragma unroll
      for (int t = 0; t < NT; ++t) full = tiles(t) > full ? tiles(t) : full;
      const int per = (full + S - 1) / S;
      kt0 = sp * per;
      kt1 = kt0 + per < full ? kt0 + per : full;
    }
    nmax = 0;
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      n_t[t] = tiles_in_range(t);
      nmax = n_t[t] > nmax ? n_t[t] : nmax;
    }
  }
  // key tiles that query tile t needs from key tile 0 on (computed, not indexed: t need not be a constant)
  __device__ __forceinline__ int tiles(int t) const {
    if (t >= n_valid) return 0;
    if (!CAUSAL) return nk;
    const int diag = q_row0 / 128 + t + 1;
    return diag < nk ? diag : nk;
  }
  // key tiles of the item's range [kt0, kt1) that query tile t needs
  __device__ __forceinline__ int tiles_in_range(int t) const {
    if constexpr (!SPLIT) return tiles(t);
    const int end = tiles(t) < kt1 ? tiles(t) : kt1;
    return end > kt0 ? end - kt0 : 0;
  }
};

template <bool BF16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  if constexpr (BF16) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
  } else {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
  }
}

// x rounded to the dtype (round to nearest even) and back to fp32.
template <bool BF16>
__device__ __forceinline__ float round_dtype(float x) {
  if constexpr (BF16) {
    return __bfloat162float(__float2bfloat16_rn(x));
  } else {
    return __half2float(__float2half_rn(x));
  }
}

// Rounds (a, b) to a packed dtype pair and returns the packed pair of the rounding residuals.
template <bool BF16>
__device__ __forceinline__ uint32_t pack2_residual(float a, float b, uint32_t& rounded) {
  rounded = pack2<BF16>(a, b);
  float ra, rb;
  if constexpr (BF16) {
    const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&rounded));
    ra = f.x;
    rb = f.y;
  } else {
    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&rounded));
    ra = f.x;
    rb = f.y;
  }
  return pack2<BF16>(a - ra, b - rb);
}

// where-codes for timeouts
enum : uint32_t {
  W_Q = 1, W_RING_EMPTY = 2, W_RING_FULL = 3, W_P = 4, W_S = 5, W_O = 6, W_DRAIN = 7,
  W_QFREE = 8, W_CLC = 9, W_ITEM = 10, W_OFREE = 11, W_SFREE = 12, W_PV = 13,
  B_CLC_ID = 20  // where-code for FA_DEV_BAD_INDEX
};

// SPLIT: the item is one of kv_splits ranges of its block's key tiles and writes a partial O and LSE
// (a separate instantiation, so the plain forward carries none of it).
template <int D, bool BF16, bool CAUSAL, bool SPLIT>
__global__ void __launch_bounds__(FwdCfg<D>::THREADS, 1) fa_fwd_kernel(const __grid_constant__ FwdParams p) {
  using C = FwdCfg<D>;
  using Item = FwdItem<C::NT, CAUSAL, SPLIT>;
  // d = 256 without a split: a launch index (x, y) is first mapped through the backward's launch order
  // (fa_bwd_order.cuh; K and V of a head are 4 N d bytes), so the items in flight share a few heads' K
  // and V in L2 (its two-slot K/V ring makes it wait on every load); every role maps its own first
  // item, and the producer maps each taken-over id before it queues it. (d = 64 and 128 measured no
  // gain from it.)
  auto item_order = [&](int& x, int& y) {
    if constexpr (!SPLIT && D == 256) bwd_block_order(x, y, gridDim.x, gridDim.y, 4ll * p.N * D, x, y);
  };
  constexpr int NT = C::NT;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sQ = smem_u32(smem);
  const uint32_t sRing = sQ + C::SMEM_Q;
  uint8_t* aux = smem + C::SMEM_Q + C::SMEM_RING;
  uint64_t* bars = reinterpret_cast<uint64_t*>(aux);
  const uint32_t b_q = smem_u32(&bars[0]);
  const uint32_t b_qfree = smem_u32(&bars[1]);
  auto b_full = [&](int s) { return smem_u32(&bars[2 + s]); };
  auto b_empty = [&](int s) { return smem_u32(&bars[2 + C::NS + s]); };
  auto b_s = [&](int t) { return smem_u32(&bars[2 + 2 * C::NS + t]); };
  auto b_p = [&](int t) { return smem_u32(&bars[2 + 2 * C::NS + NT + t]); };
  auto b_o = [&](int t) { return smem_u32(&bars[2 + 2 * C::NS + 2 * NT + t]); };
  auto b_ofree = [&](int t) { return smem_u32(&bars[2 + 2 * C::NS + 3 * NT + t]); };
  const uint32_t b_clc = smem_u32(&bars[2 + 2 * C::NS + 4 * NT]);
  auto b_item_full = [&](int i) { return smem_u32(&bars[3 + 2 * C::NS + 4 * NT + i]); };
  auto b_item_empty = [&](int i) { return smem_u32(&bars[5 + 2 * C::NS + 4 * NT + i]); };
  const uint32_t b_drain = smem_u32(&bars[7 + 2 * C::NS + 4 * NT]);
  auto b_sfree = [&](int t) { return smem_u32(&bars[8 + 2 * C::NS + 4 * NT + t]); };    // SEP_P: S_t read
  auto b_pv = [&](int t) { return smem_u32(&bars[8 + 2 * C::NS + 5 * NT + t]); };       // SEP_P: P_t V done
  const uint32_t clc_resp = smem_u32(aux + C::BAR_BYTES);
  volatile int* items = reinterpret_cast<volatile int*>(aux + C::BAR_BYTES + 16);  // [2][2]: x, y (x < 0: none)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(aux + C::BAR_BYTES + 32);
  volatile uint32_t* abort_flag = tmem_slot + 1;

  const int warp = threadIdx.x >> 5;
  const int N = p.N;

  if (threadIdx.x == 0) {
    mbar_init(b_q, 1);
    mbar_init(b_qfree, 1);
    for (int s = 0; s < C::NS; ++s) {
      mbar_init(b_full(s), 1);
      mbar_init(b_empty(s), 1);
    }
    for (int t = 0; t < NT; ++t) {
      mbar_init(b_s(t), 1);
      mbar_init(b_p(t), 128);
      mbar_init(b_o(t), 1);
      mbar_init(b_ofree(t), 128);
    }
    mbar_init(b_clc, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(b_item_full(i), 1);
      mbar_init(b_item_empty(i), 1 + 4 * NT);  // the MMA thread and one lane per softmax warp
    }
    mbar_init(b_drain, 1);
    if constexpr (C::SEP_P) {
      for (int t = 0; t < NT; ++t) {
        mbar_init(b_sfree(t), 128);
        mbar_init(b_pv(t), 1);
      }
    }
    *abort_flag = 0u;
    mbar_fence_init();
    fence_proxy_async_smem();
  }
  if (warp == 4 * NT + 1) {
    tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // Work loop shared by all roles. The CTA starts with the item it was launched
  // for; the producer then takes over not-yet-launched CTAs one at a time
  // (cluster launch control, asked while the current item's last K/V tiles are
  // loaded) and passes their ids to the other roles through a two-entry queue in
  // shared memory. An id x < 0 ends the loop. Barrier phases run on per-role
  // counters across items, so nothing is re-initialised between items.
  // Each role changes its register budget (NT = 2) and ends with its own copy of
  // the teardown barrier, so no code is shared between the two budgets.
  if (warp == 4 * NT) {
    // ------------------------------------------------------------ producer
    if constexpr (NT == 2) setmaxnreg_dec<C::OTHER_REGS>();
    if (elect_one()) {
      tma_prefetch_desc(&p.tm_q);
      tma_prefetch_desc(&p.tm_k);
      tma_prefetch_desc(&p.tm_v);
      int ix = blockIdx.x, iy = blockIdx.y;
      item_order(ix, iy);
      uint32_t seq = 0;      // K/V loads issued (ring position)
      int n_items = 0;       // items whose loads were issued
      bool clc_live = true;  // no "nothing left" answer yet
      bool clc_pending = false;
      uint32_t clc_phase = 0;
      bool ok = true;
      while (ok) {
        const Item w(ix, iy, p);
        // Q_t of the previous item is dead once its last S MMA has completed
        if (n_items > 0 && !wait_bar(b_qfree, (n_items - 1) & 1, p.timeout_ns, abort_flag, W_QFREE)) break;
        mbar_arrive_expect_tx(b_q, w.n_valid * C::TILE);
        for (int t = 0; t < w.n_valid; ++t)
#pragma unroll
          for (int c = 0; c < C::NCHUNK; ++c)
            tma_load_3d(sQ + t * C::TILE + c * C::CHUNK, &p.tm_q, b_q, c * 64, w.q_row0 + t * 128, w.bh);
        ++n_items;
        const int nload = 2 * w.nmax;
        const int ask_at = nload >= 2 ? nload - 2 : 0;  // with the item's last K/V pair (at once if it has none)
        if (SPLIT && nload == 0 && clc_live) {
          fence_proxy_async_smem();
          mbar_arrive_expect_tx(b_clc, 16);
          clc_try_cancel(clc_resp, b_clc);
          clc_pending = true;
        }
        for (int s = 0; s < nload; ++s) {
          if (s == ask_at && clc_live) {
            fence_proxy_async_smem();  // earlier generic reads of the answer slot come first
            mbar_arrive_expect_tx(b_clc, 16);
            clc_try_cancel(clc_resp, b_clc);
            clc_pending = true;
          }
          const uint32_t slot = seq % C::NS, use = seq / C::NS;
          if (use > 0 && !wait_bar(b_empty(slot), (use - 1) & 1, p.timeout_ns, abort_flag, W_RING_EMPTY)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(b_full(slot), C::TILE);
          const void* map = (s & 1) ? static_cast<const void*>(&p.tm_v) : static_cast<const void*>(&p.tm_k);
          const int krow = ((SPLIT ? w.kt0 : 0) + (s >> 1)) * 128;  // rows past N arrive as zeros
#pragma unroll
          for (int c = 0; c < C::NCHUNK; ++c)
            tma_load_3d(sRing + slot * C::TILE + c * C::CHUNK, map, b_full(slot), c * 64, krow, w.bkv);
          ++seq;
        }
        if (!ok) break;
        int nx = -1, ny = 0;
        if (clc_live) {
          if (!wait_bar(b_clc, clc_phase, p.timeout_ns, abort_flag, W_CLC)) break;
          clc_pending = false;
          clc_phase ^= 1u;
          if (!clc_query(clc_resp, nx, ny)) {
            clc_live = false;
            nx = -1;
          } else if (nx < 0 || ny < 0 || nx >= static_cast<int>(gridDim.x) || ny >= static_cast<int>(gridDim.y)) {
            // a taken-over CTA must be one of this grid's: anything else ends the CTA's work
            report_status(FA_DEV_BAD_INDEX, B_CLC_ID);
            clc_live = false;
            nx = -1;
          } else {
            item_order(nx, ny);  // the queue holds mapped ids
          }
        }
        const int qi = n_items - 1;  // queue entry qi names the item after item qi
        if (qi >= 2 && !wait_bar(b_item_empty(qi & 1), ((qi >> 1) - 1) & 1, p.timeout_ns, abort_flag, W_ITEM)) break;
        items[2 * (qi & 1)] = nx;
        items[2 * (qi & 1) + 1] = ny;
        mbar_arrive(b_item_full(qi & 1));  // release: readers acquire through their wait
        if (nx < 0) break;
        ix = nx;
        iy = ny;
      }
      // Drain: every issued copy must have landed before the CTA may exit.
      if (clc_pending) wait_bar(b_clc, clc_phase, p.timeout_ns, abort_flag, W_DRAIN);
      for (uint32_t s = (seq > C::NS ? seq - C::NS : 0u); s < seq; ++s)
        wait_bar(b_full(s % C::NS), (s / C::NS) & 1, p.timeout_ns, abort_flag, W_DRAIN);
      if (n_items > 0) wait_bar(b_q, (n_items - 1) & 1, p.timeout_ns, abort_flag, W_DRAIN);
    }
    __syncwarp();
    __syncthreads();
  } else if (warp == 4 * NT + 1) {
    // ------------------------------------------------------------ MMA issuer
    if constexpr (NT == 2) setmaxnreg_dec<C::OTHER_REGS>();
    if (elect_one()) {
      constexpr uint32_t idesc_s = make_idesc(128, 128, BF16, false, false);
      constexpr uint32_t idesc_pv = make_idesc(128, D, BF16, false, true);
      // Descriptors are built once; an MMA only adds (byte offset >> 4) to the start-address
      // field, which cannot carry out of its 14 bits because shared memory ends below 256 KB.
      const uint64_t dq0 = make_sdesc(sQ, 16, 1024);           // Q_t, K-major
      const uint64_t dk0 = make_sdesc(sRing, 16, 1024);        // K in a ring slot, K-major
      const uint64_t dv0 = make_sdesc(sRing, C::CHUNK, 1024);  // V in a ring slot, MN-major
      int ix = blockIdx.x, iy = blockIdx.y;
      item_order(ix, iy);
      uint32_t seq = 0;        // ring position of the item's K_0
      uint32_t n_p[NT] = {};   // P_t tiles consumed
      uint32_t n_o[NT] = {};   // items in which tile t produced an output
      uint32_t n_si[NT] = {};  // S_t tiles issued (SEP_P)
      int n_items = 0;
      bool ok = true;
      while (ok) {
        const Item w(ix, iy, p);
        if (!wait_bar(b_q, n_items & 1, p.timeout_ns, abort_flag, W_Q)) break;
        for (int j = 0; ok && j <= w.nmax; ++j) {
          const uint32_t sK = seq + 2 * j, sV = seq + 2 * j - 1;
          if (j > 0 && !wait_bar(b_full(sV % C::NS), (sV / C::NS) & 1, p.timeout_ns, abort_flag, W_RING_FULL)) break;
          if (j < w.nmax && !wait_bar(b_full(sK % C::NS), (sK / C::NS) & 1, p.timeout_ns, abort_flag, W_RING_FULL))
            break;
          tc_fence_after();
          if constexpr (C::SEP_P) {
            // S_t(j) first, each once the softmax has read S_t's previous tile (P has its own
            // columns), then P_t(j-1) V for each tile as its P is ready
#pragma unroll
            for (int t = 0; t < NT; ++t) {
              if (j < w.n_t[t]) {
                if (n_si[t] > 0 &&
                    !wait_bar(b_sfree(t), (n_si[t] - 1) & 1, p.timeout_ns, abort_flag, W_SFREE)) {
                  ok = false;
                  break;
                }
                ++n_si[t];
                tc_fence_after();
                const uint64_t dk = dk0 + static_cast<uint64_t>(((sK % C::NS) * C::TILE) >> 4);
                const uint64_t dq = dq0 + static_cast<uint64_t>((t * C::TILE) >> 4);
                const uint32_t tS = tmem + C::S_COL(t);
#pragma unroll
                for (int k = 0; k < D / 16; ++k) {
                  const uint64_t off = static_cast<uint64_t>(((k >> 2) * C::CHUNK + (k & 3) * 32) >> 4);
                  mma_ss(tS, dq + off, dk + off, idesc_s, k > 0 ? 1u : 0u);
                }
                mma_commit(b_s(t));
              }
            }
            if (!ok) break;
#pragma unroll
            for (int t = 0; t < NT; ++t) {
              if (j >= 1 && j <= w.n_t[t]) {
                if (!wait_bar(b_p(t), n_p[t] & 1, p.timeout_ns, abort_flag, W_P)) {
                  ok = false;
                  break;
                }
                ++n_p[t];
                if (j == 1 && n_o[t] > 0 && !wait_bar(b_ofree(t), (n_o[t] - 1) & 1, p.timeout_ns, abort_flag, W_OFREE)) {
                  ok = false;
                  break;
                }
                tc_fence_after();
                const uint64_t dv = dv0 + static_cast<uint64_t>(((sV % C::NS) * C::TILE) >> 4);
                const uint32_t tO = tmem + C::O_COL(t), tP = tmem + C::P_COL(t);
#pragma unroll
                for (int k = 0; k < 8; ++k)
                  mma_ts(tO, tP + k * 8, dv + static_cast<uint64_t>(k * (2048 >> 4)), idesc_pv,
                         (j > 1 || k > 0) ? 1u : 0u);
                mma_commit(b_pv(t));  // P_t's columns may take the next P; O_t may be rescaled
                if (j == w.n_t[t]) {
                  mma_commit(b_o(t));
                  ++n_o[t];
                }
              }
            }
          } else {
#pragma unroll
          for (int t = 0; t < NT; ++t) {
            if (j >= 1 && j <= w.n_t[t]) {
              if (!wait_bar(b_p(t), n_p[t] & 1, p.timeout_ns, abort_flag, W_P)) {
                ok = false;
                break;
              }
              ++n_p[t];
              // the first P V of an item overwrites O_t: the previous item's epilogue must have read it
              if (j == 1 && n_o[t] > 0 && !wait_bar(b_ofree(t), (n_o[t] - 1) & 1, p.timeout_ns, abort_flag, W_OFREE)) {
                ok = false;
                break;
              }
              tc_fence_after();
              const uint64_t dv = dv0 + static_cast<uint64_t>(((sV % C::NS) * C::TILE) >> 4);
              const uint32_t tO = tmem + C::O_COL(t), tP = tmem + C::S_COL(t);
#pragma unroll
              for (int k = 0; k < 8; ++k)  // 16 keys per MMA: 16 rows of V = 2048 bytes
                mma_ts(tO, tP + k * 8, dv + static_cast<uint64_t>(k * (2048 >> 4)), idesc_pv, (j > 1 || k > 0) ? 1u : 0u);
              if (j == w.n_t[t]) {
                mma_commit(b_o(t));
                ++n_o[t];
              }
            }
            if (j < w.n_t[t]) {
              const uint64_t dk = dk0 + static_cast<uint64_t>(((sK % C::NS) * C::TILE) >> 4);
              const uint64_t dq = dq0 + static_cast<uint64_t>((t * C::TILE) >> 4);
              const uint32_t tS = tmem + C::S_COL(t);
#pragma unroll
              for (int k = 0; k < D / 16; ++k) {  // 16 head dims per MMA: 32 bytes inside a 64-wide chunk
                const uint64_t off = static_cast<uint64_t>(((k >> 2) * C::CHUNK + (k & 3) * 32) >> 4);
                mma_ss(tS, dq + off, dk + off, idesc_s, k > 0 ? 1u : 0u);
              }
              mma_commit(b_s(t));
            }
          }
          }
          if (!ok) break;
          if (j == w.nmax - 1) mma_commit(b_qfree);  // every S MMA of the item has been issued
          if (j < w.nmax) mma_commit(b_empty(sK % C::NS));
          if (j > 0) mma_commit(b_empty(sV % C::NS));
        }
        if (!ok) break;
        if (SPLIT && w.nmax == 0) mma_commit(b_qfree);  // an empty key range: nothing reads Q
        seq += 2 * w.nmax;
        const int qi = n_items++;
        if (!wait_bar(b_item_full(qi & 1), (qi >> 1) & 1, p.timeout_ns, abort_flag, W_ITEM)) break;
        const int nx = items[2 * (qi & 1)], ny = items[2 * (qi & 1) + 1];
        mbar_arrive(b_item_empty(qi & 1));
        if (nx < 0) break;
        ix = nx;
        iy = ny;
      }
      // Drain: all issued MMAs complete before teardown.
      mma_commit(b_drain);
      wait_bar(b_drain, 0, p.timeout_ns, abort_flag, W_DRAIN);
    }
    __syncwarp();
    tc_fence_before();
    __syncthreads();  // every role is done with TMEM
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  } else if (warp < 4 * NT) {
    // ------------------------------------------------------------ softmax + epilogue
    if constexpr (NT == 2) setmaxnreg_inc<C::SOFTMAX_REGS>();
    const int t = warp >> 2;
    const int r = threadIdx.x & 127;  // row within the query tile == TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_off + C::S_COL(t);
    const uint32_t tO = tmem + lane_off + C::O_COL(t);
    const uint32_t tP = C::SEP_P ? tmem + lane_off + C::P_COL(t) : tS;
    const float sl2 = p.scale_log2;
    int ix = blockIdx.x, iy = blockIdx.y;
    item_order(ix, iy);
    uint32_t n_s = 0;  // S_t tiles consumed
    uint32_t n_o = 0;  // outputs written
    int n_items = 0;
    bool ok = true;
    while (ok) {
      const Item w(ix, iy, p);
      const int my_n = w.tiles_in_range(t);  // computed: t is not a compile-time index
      const int q_row = w.q_row0 + t * 128 + r;  // within the head
      // keys this row may see: those that exist, and (causal) none past the query itself
      const int klim = (CAUSAL && w.klen > q_row + 1) ? q_row + 1 : w.klen;
      float m_used = 0.f, l = 0.f;
      float l_fix = 0.f;  // sum over tiles of round(p_max) - p_max, the rounding of each tile's largest P
      for (int j = 0; ok && j < my_n; ++j) {
        // warp-uniform outcome: tcgen05.ld/st below are warp-collective
        if (!__all_sync(0xffffffffu, wait_bar(b_s(t), n_s & 1, p.timeout_ns, abort_flag, W_S))) {
          ok = false;
          break;
        }
        ++n_s;
        tc_fence_after();
        float s[128];
        {
          uint32_t u[128];
          tmem_ld128(tS, u);  // the whole row in one TMEM round trip
#pragma unroll
          for (int i = 0; i < 128; ++i) s[i] = __uint_as_float(u[i]);
        }
        if constexpr (C::SEP_P) {  // S_t may take the next tile's scores now
          tc_fence_before();
          mbar_arrive(b_sfree(t));
        }
        // SEP_P: P_t's columns and O_t are the previous P_t V's until it completes (S_t no longer
        // announces it); wait for it before the rescale or the P store, whichever comes first
        bool pv_seen = !C::SEP_P || n_s < 2;
        auto wait_pv = [&]() -> bool {
          if (pv_seen) return true;
          pv_seen = true;
          if (!__all_sync(0xffffffffu, wait_bar(b_pv(t), (n_s - 2) & 1, p.timeout_ns, abort_flag, W_PV))) return false;
          tc_fence_after();
          return true;
        };
        // keys this row may not see: past the query itself (causal, diagonal tile), past the end of
        // the sequence or past the batch's key count (last tiles); all 128 of them only for a row
        // that sees no key at all (key count 0)
        const int lim = klim - ((SPLIT ? w.kt0 : 0) + j) * 128;
        if (__any_sync(0xffffffffu, lim < 128)) {
#pragma unroll
          for (int c = 0; c < 128; ++c) s[c] = c >= lim ? -INFINITY : s[c];
        }
        float ls0 = 0.f, ls1 = 0.f;
        uint32_t pk[64];
        // P = 2^(s * scale * log2 e - m_used), its row sum, and (TRACK) the row max of s on the side
        auto exp_pass = [&](auto track) -> float {
          constexpr bool TRACK = decltype(track)::value;
          // pairs of columns go through the two-wide fp32 FMA and add (each lane of the pair rounds
          // as the scalar instruction would), which halves those instructions in this issue-bound loop
          const float2 sl2_2 = make_float2(sl2, sl2), neg_m2 = make_float2(-m_used, -m_used);
          float mx0 = -INFINITY, mx1 = -INFINITY, mx2 = -INFINITY, mx3 = -INFINITY;
          float2 ls = make_float2(0.f, 0.f);  // .x: even columns, .y: odd columns
#pragma unroll
          for (int c = 0; c < 128; c += 8) {
            float2 x[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) x[e] = __ffma2_rn(make_float2(s[c + 2 * e], s[c + 2 * e + 1]), sl2_2, neg_m2);
            if constexpr (TRACK) {
              mx0 = max3f(mx0, x[0].x, x[0].y);
              mx1 = max3f(mx1, x[1].x, x[1].y);
              mx2 = max3f(mx2, x[2].x, x[2].y);
              mx3 = max3f(mx3, x[3].x, x[3].y);
            }
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float2 pp = make_float2(ex2_approx(x[e].x), ex2_approx(x[e].y));
              ls = __fadd2_rn(ls, pp);
              pk[(c >> 1) + e] = pack2<BF16>(pp.x, pp.y);
            }
          }
          ls0 = ls.x;
          ls1 = ls.y;
          return fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3));  // max of s * sl2 - m_used
        };
        if (j == 0) {
          // first key tile: the row max comes first (two new values per three-input max, four chains)
          float mx0 = -INFINITY, mx1 = -INFINITY, mx2 = -INFINITY, mx3 = -INFINITY;
#pragma unroll
          for (int c = 0; c < 128; c += 8) {
            mx0 = max3f(mx0, s[c + 0], s[c + 1]);
            mx1 = max3f(mx1, s[c + 2], s[c + 3]);
            mx2 = max3f(mx2, s[c + 4], s[c + 5]);
            mx3 = max3f(mx3, s[c + 6], s[c + 7]);
          }
          m_used = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3)) * sl2;
          if (m_used == -INFINITY) m_used = 0.f;  // no visible key: every P is 0, l stays 0
          exp_pass(std::false_type{});
        } else {
          // later tiles: exponentiate against the running max and find the new row max on the way;
          // only a row whose max grew by more than the threshold redoes the pass
          const float x_max = exp_pass(std::true_type{});  // the tile's largest exponent against m_used
          const float m_new = x_max + m_used;
          const bool rescale = m_new > m_used + p.rescale_threshold;
          if (__any_sync(0xffffffffu, rescale)) {
            if constexpr (C::SEP_P) {
              if (!wait_pv()) {
                ok = false;
                break;
              }
            }
            const float alpha = rescale ? ex2_approx(m_used - m_new) : 1.f;
            if (rescale) {
              m_used = m_new;
              l *= alpha;
              l_fix *= alpha;
            }
            // O_t is quiescent: the commit that announced S_t(j) also covers P_t(j-1) V (or, SEP_P,
            // that product has been waited for above)
#pragma unroll 1
            for (int c = 0; c < D / 32; ++c) {
              uint32_t u[32];
              tmem_ld32(tO + 32 * c, u);
#pragma unroll
              for (int i = 0; i < 32; ++i) u[i] = __float_as_uint(__uint_as_float(u[i]) * alpha);
              tmem_st32(tO + 32 * c, u);
            }
            exp_pass(std::false_type{});
          }
          // a row that moved its max has P = 1 exactly at the tile's maximum; a row whose tile maximum
          // stayed at or below m_used holds no row-dominant weight in this tile; the rest have their
          // largest P = 2^x_max (0 < x_max <= 8), as the pass computed it
          if (!rescale && x_max > 0.f) {
            const float p_max = ex2_approx(x_max);
            l_fix += round_dtype<BF16>(p_max) - p_max;
          }
        }
        l += ls0 + ls1;
        if constexpr (C::SEP_P) {
          if (!wait_pv()) {
            ok = false;
            break;
          }
        }
        tmem_st64(tP, pk);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(b_p(t));
      }
      if (ok && my_n > 0) {
        // ---------------------------------------------------------- epilogue of tile t
        ok = __all_sync(0xffffffffu, wait_bar(b_o(t), n_o & 1, p.timeout_ns, abort_flag, W_O));
        ++n_o;
        const bool row_ok = q_row < N;  // the tile's rows past N are computed, not stored
        const size_t grow = static_cast<size_t>(w.row_base) + q_row;
        if (ok) {
          tc_fence_after();
          const float l_o = l + l_fix;  // the sum of the weights that P V used, to fp32 accuracy
          const float inv_l = l_o > 0.f ? 1.f / l_o : 0.f;  // a row with no visible key: O = 0
          // a split key range writes its normalised partial O in fp32 (and its LSE) for the merge
          constexpr bool part = SPLIT;
          const size_t prow = static_cast<size_t>(w.sp) * p.part_rows + grow;
          uint4* o_row = (p.o32 || part) ? nullptr : reinterpret_cast<uint4*>(p.o + grow * D);
          float4* o32_row = part ? reinterpret_cast<float4*>(p.part_o + prow * D)
                                 : (p.o32 ? reinterpret_cast<float4*>(p.o32 + grow * D) : nullptr);
          uint4* lo_row = (p.o_lo && !part) ? reinterpret_cast<uint4*>(p.o_lo + grow * D) : nullptr;
          constexpr int EC = D < 128 ? D : 128;  // columns per TMEM round trip
#pragma unroll 1
          for (int c0 = 0; c0 < D; c0 += EC) {
            uint32_t u[EC];
            if constexpr (EC == 128)
              tmem_ld128(tO + c0, u);
            else
              tmem_ld64(tO + c0, u);
            if (c0 + EC == D) {
              // O_t is in registers: the next item's first P V may overwrite it
              tc_fence_before();
              mbar_arrive(b_ofree(t));
            }
#pragma unroll
            for (int g = 0; g < EC / 8; ++g) {
              float x[8];
#pragma unroll
              for (int e = 0; e < 8; ++e) x[e] = __uint_as_float(u[8 * g + e]) * inv_l;
              if (o32_row) {
                if (row_ok) {
                  o32_row[2 * ((c0 >> 3) + g)] = make_float4(x[0], x[1], x[2], x[3]);
                  o32_row[2 * ((c0 >> 3) + g) + 1] = make_float4(x[4], x[5], x[6], x[7]);
                }
                continue;
              }
              uint4 v, lo;
              lo.x = pack2_residual<BF16>(x[0], x[1], v.x);
              lo.y = pack2_residual<BF16>(x[2], x[3], v.y);
              lo.z = pack2_residual<BF16>(x[4], x[5], v.z);
              lo.w = pack2_residual<BF16>(x[6], x[7], v.w);
              if (row_ok) {
                o_row[(c0 >> 3) + g] = v;
                if (lo_row) lo_row[(c0 >> 3) + g] = lo;
              }
            }
          }
          // LSE in natural log: (m_used + log2 l) * ln 2 (-inf for a row with no visible key)
          if (row_ok) (part ? p.part_lse + prow : p.lse + grow)[0] = (m_used + log2f(l)) * 0.69314718055994531f;
        }
      } else if (SPLIT && ok && q_row < N) {
        // a split key range that holds none of this tile's keys: an empty part (weight 0 in the merge)
        const size_t prow = static_cast<size_t>(w.sp) * p.part_rows + static_cast<size_t>(w.row_base) + q_row;
        float4* dst = reinterpret_cast<float4*>(p.part_o + prow * D);
#pragma unroll 4
        for (int c = 0; c < D / 4; ++c) dst[c] = make_float4(0.f, 0.f, 0.f, 0.f);
        p.part_lse[prow] = -INFINITY;
      }
      if (!ok) break;
      const int qi = n_items++;
      if (!__all_sync(0xffffffffu, wait_bar(b_item_full(qi & 1), (qi >> 1) & 1, p.timeout_ns, abort_flag, W_ITEM)))
        break;
      const int nx = items[2 * (qi & 1)], ny = items[2 * (qi & 1) + 1];
      __syncwarp();
      if ((threadIdx.x & 31) == 0) mbar_arrive(b_item_empty(qi & 1));
      if (nx < 0) break;
      ix = nx;
      iy = ny;
    }
    tc_fence_before();
    __syncthreads();
  } else {
    // ------------------------------------------------------------ idle warps of the last warpgroup
    if constexpr (NT == 2) setmaxnreg_dec<C::OTHER_REGS>();
    __syncthreads();
  }
}

// Joins the split key ranges of a query row (the online-softmax update of page
// "transformer模型详解（十）：FlashAttention优化技术", section "Tiling 分块策略", applied
// across ranges): LSE = ln sum_s e^(LSE_s), O = sum_s e^(LSE_s - LSE) O_s; a part
// with LSE_s = -inf weighs 0, and a row whose parts are all empty gets O = 0,
// LSE = -inf. One warp per row, lane l holding columns 4l .. 4l+3 (+128 for
// d = 256); O is written in the dtype (with its rounding residual when o_lo is
// given) or in fp32.
template <int D, bool BF16>
__global__ void __launch_bounds__(256) fa_fwd_merge_kernel(const float* __restrict__ part_o,
                                                            const float* __restrict__ part_lse, long long rows,
                                                            int n_split, uint16_t* o, uint16_t* o_lo, float* o32,
                                                            float* lse) {
  constexpr int V = D / 128 > 0 ? D / 128 : 1;  // float4 vectors per lane (d = 64: half the lanes)
  const int lane = threadIdx.x & 31;
  const long long warps = static_cast<long long>(gridDim.x) * (blockDim.x >> 5);
  for (long long row = static_cast<long long>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5); row < rows;
       row += warps) {
    float m = -INFINITY;
    for (int s = 0; s < n_split; ++s) m = fmaxf(m, __ldg(part_lse + s * rows + row));
    float acc[4 * V] = {};
    float wsum = 0.f;
    if (m != -INFINITY) {
      for (int s = 0; s < n_split; ++s) {
        const float ls = __ldg(part_lse + s * rows + row);
        if (ls == -INFINITY) continue;
        const float wgt = __expf(ls - m);
        wsum += wgt;
        const float4* src = reinterpret_cast<const float4*>(part_o + (s * rows + row) * D);
#pragma unroll
        for (int v = 0; v < V; ++v) {
          if (D == 64 && lane >= 16) break;
          const float4 x = __ldg(src + lane + 32 * v);
          acc[4 * v] += wgt * x.x;
          acc[4 * v + 1] += wgt * x.y;
          acc[4 * v + 2] += wgt * x.z;
          acc[4 * v + 3] += wgt * x.w;
        }
      }
    }
    const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
#pragma unroll
    for (int v = 0; v < V; ++v) {
      if (D == 64 && lane >= 16) break;
      const float x0 = acc[4 * v] * inv, x1 = acc[4 * v + 1] * inv, x2 = acc[4 * v + 2] * inv,
                  x3 = acc[4 * v + 3] * inv;
      const long long e = row * D + 4 * (lane + 32 * v);
      if (o32) {
        *reinterpret_cast<float4*>(o32 + e) = make_float4(x0, x1, x2, x3);
      } else {
        uint2 r, lo;
        lo.x = pack2_residual<BF16>(x0, x1, r.x);
        lo.y = pack2_residual<BF16>(x2, x3, r.y);
        *reinterpret_cast<uint2*>(o + e) = r;
        if (o_lo) *reinterpret_cast<uint2*>(o_lo + e) = lo;
      }
    }
    if (lane == 0) lse[row] = wsum > 0.f ? m + __logf(wsum) : -INFINITY;
  }
}

template <int D, bool BF16, bool CAUSAL, bool SPLIT>
cudaError_t launch_fwd_t(const FwdArgs& a) {
  using C = FwdCfg<D>;
  auto kern = fa_fwd_kernel<D, BF16, CAUSAL, SPLIT>;
  static std::atomic<unsigned long long> attr_done{0};
  cudaError_t e = smem_attr_once(reinterpret_cast<const void*>(kern), C::SMEM_BYTES, attr_done);
  if (e != cudaSuccess) return e;
  if constexpr (C::NT == 2) {
    static int checked = 0;  // 1: the compiled register count matches the split
    if (!checked) {
      cudaFuncAttributes fa_attr;
      if ((e = cudaFuncGetAttributes(&fa_attr, kern)) != cudaSuccess) return e;
      if (fa_attr.numRegs != C::LAUNCH_REGS) return cudaErrorInvalidConfiguration;
      checked = 1;
    }
  }
  FwdParams p;
  p.tm_q = a.tm_q;
  p.tm_k = a.tm_k;
  p.tm_v = a.tm_v;
  p.o = a.o_f32 ? nullptr : static_cast<uint16_t*>(a.o);
  p.o32 = a.o_f32 ? static_cast<float*>(a.o) : nullptr;
  p.lse = a.lse;
  p.o_lo = static_cast<uint16_t*>(a.o_lo);
  p.kv_len = a.kv_len;
  p.kv_splits = a.kv_splits > 1 ? a.kv_splits : 1;
  p.part_o = a.part_o;
  p.part_lse = a.part_lse;
  p.part_rows = static_cast<long long>(a.B) * a.H * a.N;
  p.N = a.N;
  p.H = a.H;
  p.G = a.H / a.Hkv;
  p.tpi = (a.tiles_per_item >= 1 && a.tiles_per_item < C::NT && !SPLIT) ? a.tiles_per_item : C::NT;
  p.n_qblk = (a.N + 128 * p.tpi - 1) / (128 * p.tpi);
  p.scale_log2 = a.scale * 1.4426950408889634f;
  p.rescale_threshold = 8.0f;
  p.timeout_ns = a.timeout_ns;
  dim3 grid(a.B * a.H, p.n_qblk * p.kv_splits, 1);
  e = launch_kernel(kern, grid, dim3(C::THREADS), C::SMEM_BYTES, a.stream, p);
  if (e != cudaSuccess || p.kv_splits == 1) return e;
  const long long blocks_needed = (p.part_rows + 7) / 8;  // 8 rows (warps) per block
  const int blocks = static_cast<int>(blocks_needed < 152 * 16 ? blocks_needed : 152 * 16);
  return launch_kernel(fa_fwd_merge_kernel<D, BF16>, dim3(blocks), dim3(256), 0, a.stream,
                       static_cast<const float*>(a.part_o), static_cast<const float*>(a.part_lse), p.part_rows,
                       p.kv_splits, p.o, p.o_lo, p.o32, a.lse);
}

}  // namespace

cudaError_t launch_fwd(const FwdArgs& a) {
#define FA_FWD_CASE(D_, S_)                                                                          \
  if (a.d == D_) {                                                                                   \
    if (a.bf16) return a.causal ? launch_fwd_t<D_, true, true, S_>(a) : launch_fwd_t<D_, true, false, S_>(a); \
    return a.causal ? launch_fwd_t<D_, false, true, S_>(a) : launch_fwd_t<D_, false, false, S_>(a);          \
  }
  if (a.kv_splits > 1) {
    FA_FWD_CASE(64, true)
    FA_FWD_CASE(128, true)
    FA_FWD_CASE(256, true)
  } else {
    FA_FWD_CASE(64, false)
    FA_FWD_CASE(128, false)
    FA_FWD_CASE(256, false)
  }
#undef FA_FWD_CASE
  return cudaErrorInvalidValue;
}

cudaError_t read_clear_status_fwd(DevStatusHost* out, cudaStream_t s) {
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
