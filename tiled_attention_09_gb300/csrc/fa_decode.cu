// Paged decode attention for sm_103a: split-key partial attention (K5) and the split merge (K6).
//
// Method. A few new queries per sequence (Mq of them, the last Mq positions) attend to a long
// key/value history kept in fixed-size pages. Page "高级特性：探索PyTorch/XLA的Pallas内核和Flash
// Attention实现", section "Pallas内核：自定义高效计算的关键", names such a kernel: paged attention
// for the multi-query case, K/V heads shared by several query heads. The arithmetic per query is
// the forward's online softmax (page "transformer模型详解（十）：FlashAttention优化技术", section
// "Tiling 分块策略": per key tile the local max and exponential sum, a rescale of the running sum
// and output, one normalisation at the end). The key range is cut into splits processed by
// different CTAs; each produces, per query row, an output O_s normalised by its own sum and its
// log-sum-exp LSE_s. The merge is the same online-softmax update applied across the splits:
//   LSE = ln sum_s exp(LSE_s),   O = sum_s exp(LSE_s - LSE) O_s.
//
// GB300 design. Decoding reads every cached key and value once, so the kernel is bound by HBM
// bandwidth, and with G query heads per K/V head each key is used by R = G * Mq query rows. A CTA
// owns one K/V head of one sequence and one split; its R query rows (the G heads' Mq queries are
// consecutive rows of q) form one 128-row tile, so the tile's products run on the tensor core
// (tcgen05.mma, rows past R are never read back). One thread issues a tcgen05.mma only every
// ~150 cycles, so the products of a key tile are split between two issuing warps: S(j) = Q K(j)^T
// into one of two TMEM buffers (j & 1), and O += P(j) V(j) with P(j) read from that buffer. The
// S issuer computes S(j + 1) while the softmax warps turn S(j) into P(j) and while O += P(j - 1)
// V(j - 1) runs, and waits only before reusing a buffer (its previous P must have been read). The
// softmax's lazy rescale of O waits for the previous P V only when a row's max has grown.
// K and V tiles are gathered page by page with TMA into two rings of shared-memory slots, the K
// ring consumed in order by the S issuer and the V ring by the P V issuer (one in-order consumer
// per ring keeps a slot's full-barrier parity unambiguous). Pages past the sequence's end are not
// read (zero-filled), and value rows past its end inside the last tile are zeroed before use (a
// stale page tail may hold non-finite values, and 0 * NaN is NaN in the product).
// Roles (224 threads): warps 0-3 softmax (only the warps holding rows < R work), warp 4 TMA
// producer, warp 5 the S issuer (and TMEM owner), warp 6 the P V issuer.
// Tiles hold BK = 128 keys (64 for d = 256, whose 64 KB Q tile leaves room for two 32 KB slots per
// ring only at that height).
// TMEM: S buffers at 0 and 128 (fp32 128 x BK; P as 16-bit pairs over them), O at 256 (d columns).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "common.cuh"
#include "launch.h"

namespace fa {
namespace {

struct DecParams {
  CUtensorMap tm_q;        // [B*H*Mq rows][d], box {64, 128}
  CUtensorMap tm_k, tm_v;  // [Hkv][P*page_size rows][d], box {64, min(page_size, 128), 1}
  const int* page_table;   // [B][max_pages]
  const int* ctx_len;      // [B]
  float* o_part;           // [n_split][B*H*Mq][d] fp32, each split's part normalised by its own sum
  float* lse_part;         // [n_split][B*H*Mq]
  void* o_final;           // with one split: O [B*H*Mq][d] dtype and LSE written here directly
  float* lse_final;
  int direct;              // one split: no partials, no merge
  int H, G, Mq, R;         // query heads, query heads per K/V head, queries per head, rows per CTA
  int ps_log2;             // log2(page size)
  int max_pages, n_pages;  // page-table row length, pages in the cache
  int tiles_per_split;     // 128-key tiles per split
  int rows_total;          // B*H*Mq
  int causal;
  float scale_log2;
  float rescale_threshold;
  unsigned long long timeout_ns;
};

template <int D>
struct DecCfg {
  static constexpr int BK = D == 256 ? 64 : 128;   // keys per tile (d = 256: 64, so that two slots per ring fit)
  static constexpr int QCHUNK = 128 * 128;         // Q: 128 rows x 64 elements x 2 bytes
  static constexpr int CHUNK = BK * 128;           // K or V: BK rows x 64 elements x 2 bytes
  static constexpr int NCH = D / 64;
  static constexpr int QTILE = 128 * D * 2;
  static constexpr int TILE = BK * D * 2;          // one K or one V tile
  // ring slots (one K or one V tile each) filling the rest of the 227 KB, half for K, half for V
  static constexpr int NS_FIT = (227 * 1024 - 1024 - QTILE - 512) / TILE;
  static constexpr int NSR = (NS_FIT > 12 ? 12 : NS_FIT) / 2;  // slots per ring
  // q, kfull[NSR], kempty[NSR], vfull[NSR], vempty[NSR], sfull[2], pfull[2], pvdone[2], odone, drain[2]
  static constexpr int NBAR = 1 + 4 * NSR + 6 + 1 + 2;
  static constexpr int BAR_BYTES = (NBAR * 8 + 15) & ~15;
  static constexpr int SMEM_BYTES = 1024 + QTILE + 2 * NSR * TILE + BAR_BYTES + 16;
  static constexpr int THREADS = 224;
  static_assert(NSR >= 2, "a ring must hold the tile in use and the next one");
  static_assert(SMEM_BYTES <= 227 * 1024, "smem budget");
  static_assert(256 + D <= 512, "TMEM budget");  // S buffers at 0 and 128 (BK columns each), O at 256
};

template <bool BF16>
__device__ __forceinline__ uint32_t dpack2(float lo, float hi) {
  if constexpr (BF16) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
  } else {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
  }
}

enum : uint32_t {
  WD_Q = 31, WD_EMPTY = 32, WD_FULL = 33, WD_P = 34, WD_S = 35, WD_O = 36, WD_V = 37, WD_DRAIN = 38, WD_PV = 39
};

// The CTA's split of one sequence: BK-key tiles [lo, lo + n) of the sequence's ceil(ctx / BK).
template <int BK>
struct DecWork {
  int b, hk, ctx, lo, n;
  __device__ __forceinline__ DecWork(const DecParams& p) {
    const int Hkv = p.H / p.G;
    b = blockIdx.x / Hkv;
    hk = blockIdx.x - b * Hkv;
    const int cap = p.max_pages << p.ps_log2;
    const int c = __ldg(p.ctx_len + b);
    ctx = c < 0 ? 0 : (c > cap ? cap : c);
    const int n_tiles = (ctx + BK - 1) / BK;
    lo = blockIdx.y * p.tiles_per_split;
    int hi = lo + p.tiles_per_split;
    hi = hi < n_tiles ? hi : n_tiles;
    n = hi > lo ? hi - lo : 0;
  }
};

template <int D, bool BF16>
__global__ void __launch_bounds__(224, 1) fa_decode_kernel(const __grid_constant__ DecParams p) {
  using C = DecCfg<D>;
  constexpr int NSR = C::NSR, BK = C::BK;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sQ = smem_u32(smem);
  const uint32_t sK = sQ + C::QTILE;             // K ring
  const uint32_t sV = sK + NSR * C::TILE;        // V ring
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::QTILE + 2 * NSR * C::TILE);
  const uint32_t b_q = smem_u32(&bars[0]);
  auto b_kfull = [&](int s) { return smem_u32(&bars[1 + s]); };
  auto b_kempty = [&](int s) { return smem_u32(&bars[1 + NSR + s]); };
  auto b_vfull = [&](int s) { return smem_u32(&bars[1 + 2 * NSR + s]); };
  auto b_vempty = [&](int s) { return smem_u32(&bars[1 + 3 * NSR + s]); };
  auto b_sfull = [&](int b) { return smem_u32(&bars[1 + 4 * NSR + b]); };
  auto b_pfull = [&](int b) { return smem_u32(&bars[3 + 4 * NSR + b]); };
  auto b_pvdone = [&](int b) { return smem_u32(&bars[5 + 4 * NSR + b]); };
  const uint32_t b_odone = smem_u32(&bars[7 + 4 * NSR]);
  auto b_drain = [&](int i) { return smem_u32(&bars[8 + 4 * NSR + i]); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::QTILE + 2 * NSR * C::TILE + C::BAR_BYTES);
  volatile uint32_t* abort_flag = tmem_slot + 1;

  const int warp = threadIdx.x >> 5;
  const DecWork<BK> w(p);
  const int nact = (p.R + 31) / 32;  // softmax warps that hold rows < R

  if (threadIdx.x == 0) {
    mbar_init(b_q, 1);
    for (int s = 0; s < NSR; ++s) {
      mbar_init(b_kfull(s), 1);
      mbar_init(b_kempty(s), 1);
      mbar_init(b_vfull(s), 1);
      mbar_init(b_vempty(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(b_sfull(b), 1);
      mbar_init(b_pfull(b), 32 * nact);
      mbar_init(b_pvdone(b), 1);
      mbar_init(b_drain(b), 1);
    }
    mbar_init(b_odone, 1);
    *abort_flag = 0u;
    mbar_fence_init();
    fence_proxy_async_smem();
  }
  if (warp == 5) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int q_row0 = (w.b * p.H + w.hk * p.G) * p.Mq;  // first of the CTA's R query rows
  const int n = w.n;

  if (warp == 4) {
    // ------------------------------------------------------------ producer (the whole warp)
    // A BK-key tile is BK / min(page_size, BK) page boxes per 64-column chunk; lane l issues box
    // l / NCH, chunk l % NCH, after looking up its own page, so small pages cost one round of loads.
    const int lane = threadIdx.x & 31;
    const int ps = 1 << p.ps_log2;
    const int br = ps < BK ? ps : BK;             // rows per TMA box
    const int nbox = (BK / br) * C::NCH;          // boxes per tile (at most 16)
    const int oob_row = p.n_pages << p.ps_log2;   // the first row past the cache: the box reads zeros
    const int* ptab = p.page_table + static_cast<size_t>(w.b) * p.max_pages;
    const int r0 = (lane / C::NCH) * br, cc = lane % C::NCH;  // this lane's box: first row, chunk
    if (lane == 0) {
      tma_prefetch_desc(&p.tm_q);
      tma_prefetch_desc(&p.tm_k);
      tma_prefetch_desc(&p.tm_v);
      mbar_arrive_expect_tx(b_q, C::QTILE);
#pragma unroll
      for (int c = 0; c < C::NCH; ++c) tma_load_2d(sQ + c * C::QCHUNK, &p.tm_q, b_q, c * 64, q_row0);
    }
    // tile j of the split into ring slot j % NSR
    auto load = [&](uint32_t ring, uint32_t full, uint32_t empty, const CUtensorMap* map, int j) -> bool {
      const int slot = j % NSR, use = j / NSR;
      bool ok = true;
      if (lane == 0) {
        if (use > 0) ok = wait_bar(empty + 8 * slot, (use - 1) & 1, p.timeout_ns, abort_flag, WD_EMPTY);
        if (ok) mbar_arrive_expect_tx(full + 8 * slot, C::TILE);
      }
      if (!__shfl_sync(0xffffffffu, ok, 0)) return false;
      if (lane < nbox) {
        const int key = (w.lo + j) * BK + r0;
        int y = oob_row;
        if (key < w.ctx) {  // pages wholly past the sequence are not read
          const int pid = __ldg(ptab + (key >> p.ps_log2));
          if (pid >= 0 && pid < p.n_pages) y = (pid << p.ps_log2) + (key & (ps - 1));
        }
        tma_load_3d(ring + slot * C::TILE + cc * C::CHUNK + r0 * 128, map, full + 8 * slot, cc * 64, y, w.hk);
      }
      return true;
    };
    int j = 0;
    for (; j < n; ++j)
      if (!load(sK, b_kfull(0), b_kempty(0), &p.tm_k, j) || !load(sV, b_vfull(0), b_vempty(0), &p.tm_v, j)) break;
    // Drain: every issued copy has landed before the CTA may exit.
    if (lane == 0) {
      for (int i = (j > NSR ? j - NSR : 0); i < j; ++i) {
        wait_bar(b_kfull(i % NSR), (i / NSR) & 1, p.timeout_ns, abort_flag, WD_DRAIN);
        wait_bar(b_vfull(i % NSR), (i / NSR) & 1, p.timeout_ns, abort_flag, WD_DRAIN);
      }
      wait_bar(b_q, 0, p.timeout_ns, abort_flag, WD_DRAIN);
    }
    __syncwarp();
    tc_fence_before();
    __syncthreads();
  } else if (warp == 5) {
    // ------------------------------------------------------------ S issuer: S(j) = Q K(j)^T into buffer j & 1
    if (elect_one()) {
      constexpr uint32_t idesc_s = make_idesc(128, BK, BF16, false, false);
      const uint64_t dq0 = make_sdesc(sQ, 16, 1024);  // Q, K-major
      const uint64_t dk0 = make_sdesc(sK, 16, 1024);  // K ring slot, K-major
      bool ok = wait_bar(b_q, 0, p.timeout_ns, abort_flag, WD_Q);
      for (int j = 0; ok && j < n; ++j) {
        const int slot = j % NSR, b = j & 1;
        if (!wait_bar(b_kfull(slot), (j / NSR) & 1, p.timeout_ns, abort_flag, WD_FULL)) break;
        // the buffer still holds P(j - 2) until O += P(j - 2) V(j - 2) has read it
        if (j >= 2 && !wait_bar(b_pvdone(b), ((j - 2) >> 1) & 1, p.timeout_ns, abort_flag, WD_PV)) break;
        tc_fence_after();
        const uint64_t dk = dk0 + static_cast<uint64_t>((slot * C::TILE) >> 4);
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {  // 16 head dims per MMA
          const uint64_t qo = static_cast<uint64_t>(((k >> 2) * C::QCHUNK + (k & 3) * 32) >> 4);
          const uint64_t ko = static_cast<uint64_t>(((k >> 2) * C::CHUNK + (k & 3) * 32) >> 4);
          mma_ss(tmem + 128 * b, dq0 + qo, dk + ko, idesc_s, k > 0 ? 1u : 0u);
        }
        mma_commit(b_sfull(b));
        mma_commit(b_kempty(slot));
      }
      mma_commit(b_drain(0));
      wait_bar(b_drain(0), 0, p.timeout_ns, abort_flag, WD_DRAIN);
    }
    __syncwarp();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  } else if (warp == 6) {
    // ------------------------------------------------------------ P V issuer: O += P(j) V(j)
    if (elect_one()) {
      constexpr uint32_t idesc_pv = make_idesc(128, D, BF16, false, true);
      const uint64_t dv0 = make_sdesc(sV, C::CHUNK, 1024);  // V ring slot, MN-major
      for (int j = 0; j < n; ++j) {
        const int slot = j % NSR, b = j & 1;
        if (!wait_bar(b_pfull(b), (j >> 1) & 1, p.timeout_ns, abort_flag, WD_P) ||
            !wait_bar(b_vfull(slot), (j / NSR) & 1, p.timeout_ns, abort_flag, WD_FULL))
          break;
        tc_fence_after();
        const uint64_t dv = dv0 + static_cast<uint64_t>((slot * C::TILE) >> 4);
#pragma unroll
        for (int k = 0; k < BK / 16; ++k)  // 16 keys per MMA: 16 rows of V = 2048 bytes
          mma_ts(tmem + 256, tmem + 128 * b + k * 8, dv + static_cast<uint64_t>(k * (2048 >> 4)), idesc_pv,
                 (j > 0 || k > 0) ? 1u : 0u);
        mma_commit(b_pvdone(b));
        mma_commit(b_vempty(slot));
        if (j == n - 1) mma_commit(b_odone);
      }
      mma_commit(b_drain(1));
      wait_bar(b_drain(1), 0, p.timeout_ns, abort_flag, WD_DRAIN);
    }
    __syncwarp();
    tc_fence_before();
    __syncthreads();
  } else if (warp < nact) {
    // ------------------------------------------------------------ softmax + epilogue
    const int r = threadIdx.x;  // query row of the CTA (0 .. R-1 are real) == TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
    const uint32_t tO = tmem + lane_off + 256;
    const float sl2 = p.scale_log2;
    // keys this row may see: the sequence's, and (causal) none after the query's own position
    // ctx - Mq + i, i = r % Mq
    int klim = w.ctx;
    if (p.causal) klim = w.ctx - p.Mq + (r % p.Mq) + 1;
    float m_used = 0.f, l = 0.f;
    bool ok = true;
    for (int j = 0; j < n; ++j) {
      const int b = j & 1;
      const uint32_t tS = tmem + lane_off + 128 * b;
      if (!__all_sync(0xffffffffu, wait_bar(b_sfull(b), (j >> 1) & 1, p.timeout_ns, abort_flag, WD_S))) {
        ok = false;
        break;
      }
      tc_fence_after();
      const int kt = w.lo + j;
      float s[BK];
      {
        uint32_t u[BK];
        if constexpr (BK == 128)
          tmem_ld128(tS, u);
        else
          tmem_ld64(tS, u);
#pragma unroll
        for (int i = 0; i < BK; ++i) s[i] = __uint_as_float(u[i]);
      }
      const int lim = klim - kt * BK;
      if (__any_sync(0xffffffffu, lim < BK)) {
#pragma unroll
        for (int c = 0; c < BK; ++c) s[c] = c >= lim ? -INFINITY : s[c];
      }
      float mx[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) mx[e] = -INFINITY;
#pragma unroll
      for (int c = 0; c < BK; c += 16) {
#pragma unroll
        for (int e = 0; e < 8; ++e) mx[e] = max3f(mx[e], s[c + 2 * e], s[c + 2 * e + 1]);
      }
      const float m_tile =
          fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])), fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7]))) * sl2;
      if (j == 0) {
        m_used = m_tile == -INFINITY ? 0.f : m_tile;  // no visible key yet: every P is 0
      } else {
        // lazy rescale: the running max moves only when the row max grows past the threshold; O must
        // then be quiescent, i.e. O += P(j - 1) V(j - 1) complete
        const bool rescale = m_tile > m_used + p.rescale_threshold;
        if (__any_sync(0xffffffffu, rescale)) {
          if (!__all_sync(0xffffffffu,
                          wait_bar(b_pvdone((j - 1) & 1), ((j - 1) >> 1) & 1, p.timeout_ns, abort_flag, WD_PV))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const float alpha = rescale ? ex2_approx(m_used - m_tile) : 1.f;
          if (rescale) {
            m_used = m_tile;
            l *= alpha;
          }
#pragma unroll 1
          for (int c = 0; c < D / 32; ++c) {
            uint32_t u[32];
            tmem_ld32(tO + 32 * c, u);
#pragma unroll
            for (int i = 0; i < 32; ++i) u[i] = __float_as_uint(__uint_as_float(u[i]) * alpha);
            tmem_st32(tO + 32 * c, u);
          }
        }
      }
      uint32_t pk[BK / 2];
      float ls[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) ls[e] = 0.f;
      const float neg_m = -m_used;
#pragma unroll
      for (int c = 0; c < BK; c += 2) {
        const float p0 = ex2_approx(fmaf(s[c], sl2, neg_m));
        const float p1 = ex2_approx(fmaf(s[c + 1], sl2, neg_m));
        ls[(c >> 1) & 7] += p0 + p1;
        pk[c >> 1] = dpack2<BF16>(p0, p1);
      }
      l += ((ls[0] + ls[1]) + (ls[2] + ls[3])) + ((ls[4] + ls[5]) + (ls[6] + ls[7]));
      // The sequence's last tile: value rows past its end may come from a stale page tail; zero them
      // (after their copy has landed) so that P = 0 there cannot meet a non-finite value. V(j) is load
      // j of the V ring; the slot's previous load (j - NSR <= j - 2) was consumed by O += P V before
      // S(j) could be issued, so the parity names this load's phase.
      const int valid = w.ctx - kt * BK;
      if (valid < BK) {
        const int slot = j % NSR;
        if (!__all_sync(0xffffffffu, wait_bar(b_vfull(slot), (j / NSR) & 1, p.timeout_ns, abort_flag, WD_V))) {
          ok = false;
          break;
        }
        uint8_t* vt = smem + C::QTILE + (NSR + slot) * C::TILE;
        for (int row = valid + r; row < BK; row += 32 * nact) {
#pragma unroll
          for (int c = 0; c < C::NCH; ++c) {
            uint4* z = reinterpret_cast<uint4*>(vt + c * C::CHUNK + row * 128);
#pragma unroll
            for (int u = 0; u < 8; ++u) z[u] = make_uint4(0u, 0u, 0u, 0u);
          }
        }
        fence_proxy_async_smem();  // visible to the tensor core before P is announced
      }
      if constexpr (BK == 128)
        tmem_st64(tS, pk);
      else
        tmem_st32(tS, pk);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(b_pfull(b));
    }
    // ---------------------------------------------------------- epilogue: the split's partial result
    // (with a single split, the final O in the dtype and LSE)
    const bool row_ok = r < p.R;
    if (p.direct) {
      const size_t grow = static_cast<size_t>(q_row0) + r;
      uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.o_final) + grow * D);
      bool have = false;
      if (ok && n > 0) {
        ok = __all_sync(0xffffffffu, wait_bar(b_odone, 0, p.timeout_ns, abort_flag, WD_O));
        have = ok;
      }
      if (have) {
        tc_fence_after();
        const float inv_l = l > 0.f ? 1.f / l : 0.f;
#pragma unroll 1
        for (int c0 = 0; c0 < D; c0 += 64) {
          uint32_t u[64];
          tmem_ld64(tO + c0, u);
          if (row_ok) {
#pragma unroll
            for (int g = 0; g < 8; ++g) {
              const float* x = reinterpret_cast<const float*>(u + 8 * g);
              dst[(c0 >> 3) + g] = make_uint4(dpack2<BF16>(x[0] * inv_l, x[1] * inv_l), dpack2<BF16>(x[2] * inv_l, x[3] * inv_l),
                                              dpack2<BF16>(x[4] * inv_l, x[5] * inv_l), dpack2<BF16>(x[6] * inv_l, x[7] * inv_l));
            }
          }
        }
        if (row_ok) p.lse_final[grow] = l > 0.f ? (m_used + log2f(l)) * 0.69314718055994531f : -INFINITY;
      } else if (ok && row_ok) {  // no key at all: O = 0, LSE = -inf
#pragma unroll 4
        for (int g = 0; g < D / 8; ++g) dst[g] = make_uint4(0u, 0u, 0u, 0u);
        p.lse_final[grow] = -INFINITY;
      }
      tc_fence_before();
      __syncthreads();
      return;
    }
    const size_t grow = static_cast<size_t>(blockIdx.y) * p.rows_total + q_row0 + r;
    float4* dst = reinterpret_cast<float4*>(p.o_part + grow * D);
    if (ok && n > 0) {
      ok = __all_sync(0xffffffffu, wait_bar(b_odone, 0, p.timeout_ns, abort_flag, WD_O));
      if (ok) {
        tc_fence_after();
        const float inv_l = l > 0.f ? 1.f / l : 0.f;
#pragma unroll 1
        for (int c0 = 0; c0 < D; c0 += 64) {
          uint32_t u[64];
          tmem_ld64(tO + c0, u);
          if (row_ok) {
#pragma unroll
            for (int g = 0; g < 16; ++g)
              dst[(c0 >> 2) + g] = make_float4(__uint_as_float(u[4 * g]) * inv_l, __uint_as_float(u[4 * g + 1]) * inv_l,
                                               __uint_as_float(u[4 * g + 2]) * inv_l,
                                               __uint_as_float(u[4 * g + 3]) * inv_l);
          }
        }
        if (row_ok) p.lse_part[grow] = l > 0.f ? (m_used + log2f(l)) * 0.69314718055994531f : -INFINITY;
      }
    } else if (ok && row_ok) {  // no tile in this split for the sequence: an empty partial
#pragma unroll 4
      for (int g = 0; g < D / 4; ++g) dst[g] = make_float4(0.f, 0.f, 0.f, 0.f);
      p.lse_part[grow] = -INFINITY;
    }
    tc_fence_before();
    __syncthreads();
  } else {
    // ------------------------------------------------------------ softmax warps without rows < R
    __syncthreads();
  }
}

// LSE = ln sum_s exp(LSE_s), O = sum_s exp(LSE_s - LSE) O_s, rounded to the dtype; a row whose parts
// are all empty gets O = 0 and LSE = -inf. One block per row: thread (s, cv) loads part s's 8 columns
// cv*8 .. cv*8+7 (all parts' loads in flight at once), then the weighted values are summed over the
// parts in shared memory. blockDim = VPR * NPP, NPP a power of two >= n_part.
template <int VPR, bool BF16>
__global__ void __launch_bounds__(1024) fa_decode_merge_kernel(const float4* __restrict__ o_part,
                                                               const float* __restrict__ lse_part,
                                                               uint4* __restrict__ o, float* __restrict__ lse, int rows,
                                                               int n_part) {
  extern __shared__ float sm[];
  const int npp = blockDim.x / VPR;
  float* s_lse = sm;        // [npp]
  float* s_val = sm + npp;  // [npp][VPR][9]: 8 weighted values and the weight
  const size_t row = blockIdx.x;
  const int s = threadIdx.x / VPR, cv = threadIdx.x % VPR;
  float ls = -INFINITY;
  float4 a = make_float4(0.f, 0.f, 0.f, 0.f), b = a;
  if (s < n_part) {
    ls = __ldg(lse_part + static_cast<size_t>(s) * rows + row);
    const float4* src = o_part + (static_cast<size_t>(s) * rows + row) * (VPR * 2) + 2 * cv;
    a = __ldg(src);
    b = __ldg(src + 1);
  }
  if (cv == 0) s_lse[s] = ls;
  __syncthreads();
  float m = -INFINITY;
  for (int t = 0; t < n_part; ++t) m = fmaxf(m, s_lse[t]);
  const float wgt = __expf(ls - (m == -INFINITY ? 0.f : m));  // 0 for an empty part (or no part)
  float* v = s_val + (s * VPR + cv) * 9;
  v[0] = wgt * a.x;
  v[1] = wgt * a.y;
  v[2] = wgt * a.z;
  v[3] = wgt * a.w;
  v[4] = wgt * b.x;
  v[5] = wgt * b.y;
  v[6] = wgt * b.z;
  v[7] = wgt * b.w;
  v[8] = wgt;
  __syncthreads();
  for (int half = npp / 2; half > 0; half >>= 1) {
    if (s < half) {
      const float* u = s_val + ((s + half) * VPR + cv) * 9;
#pragma unroll
      for (int k = 0; k < 9; ++k) v[k] += u[k];
    }
    __syncthreads();
  }
  if (s == 0) {
    const float wsum = v[8];
    const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
    o[row * VPR + cv] = make_uint4(dpack2<BF16>(v[0] * inv, v[1] * inv), dpack2<BF16>(v[2] * inv, v[3] * inv),
                                   dpack2<BF16>(v[4] * inv, v[5] * inv), dpack2<BF16>(v[6] * inv, v[7] * inv));
    if (cv == 0) lse[row] = wsum > 0.f ? m + logf(wsum) : -INFINITY;
  }
}

template <int D, bool BF16>
cudaError_t launch_decode_t(const DecArgs& a) {
  using C = DecCfg<D>;
  auto kern = fa_decode_kernel<D, BF16>;
  static std::atomic<unsigned long long> attr_done{0};
  cudaError_t e = smem_attr_once(reinterpret_cast<const void*>(kern), C::SMEM_BYTES, attr_done);
  if (e != cudaSuccess) return e;
  DecParams p;
  p.tm_q = a.tm_q;
  p.tm_k = a.tm_k;
  p.tm_v = a.tm_v;
  p.page_table = a.page_table;
  p.ctx_len = a.ctx_len;
  p.o_part = a.ws_o;
  p.lse_part = a.ws_lse;
  p.o_final = a.o;
  p.lse_final = a.lse;
  p.direct = a.n_split == 1 ? 1 : 0;
  p.H = a.H;
  p.G = a.H / a.Hkv;
  p.Mq = a.Mq;
  p.R = p.G * a.Mq;
  p.ps_log2 = a.ps_log2;
  p.max_pages = a.max_pages;
  p.n_pages = a.n_pages;
  p.tiles_per_split = a.tiles_per_split;
  p.rows_total = a.B * a.H * a.Mq;
  p.causal = a.causal ? 1 : 0;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  p.rescale_threshold = 8.0f;
  p.timeout_ns = a.timeout_ns;
  e = launch_kernel(kern, dim3(a.B * a.Hkv, a.n_split, 1), dim3(C::THREADS), C::SMEM_BYTES, a.stream, p);
  if (e != cudaSuccess) return e;
  if (p.direct) return cudaSuccess;
  int npp = 1;
  while (npp < a.n_split) npp <<= 1;
  const int threads = npp * (D / 8);  // n_split <= 64 (host check): at most 1024 threads
  const size_t smem = static_cast<size_t>(npp) * (1 + (D / 8) * 9) * sizeof(float);
  return launch_kernel(fa_decode_merge_kernel<D / 8, BF16>, dim3(static_cast<unsigned>(p.rows_total)), dim3(threads),
                       smem, a.stream, reinterpret_cast<const float4*>(a.ws_o), static_cast<const float*>(a.ws_lse),
                       static_cast<uint4*>(a.o), a.lse, p.rows_total, a.n_split);
}

}  // namespace

cudaError_t launch_decode(const DecArgs& a) {
  if (a.d == 256) return a.bf16 ? launch_decode_t<256, true>(a) : launch_decode_t<256, false>(a);
  if (a.d == 128) return a.bf16 ? launch_decode_t<128, true>(a) : launch_decode_t<128, false>(a);
  if (a.d == 64) return a.bf16 ? launch_decode_t<64, true>(a) : launch_decode_t<64, false>(a);
  return cudaErrorInvalidValue;
}

cudaError_t read_clear_status_decode(DevStatusHost* out, cudaStream_t s) {
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
