// C ABI of libfa.so: argument checks, TMA tensor maps, dispatch, status words.
// Declarations and the contract of every entry point are in include/fa.h.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <functional>
#include <mutex>
#include <queue>
#include <vector>

#include "../../include/fa.h"
#include "launch.h"

namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

unsigned long long g_timeout_ns = 4000000000ull;

// Tensor maps are pure functions of (base, shape, box, type); encoding one is host work on every call,
// so each host thread keeps the last few it built (direct-mapped by a hash of the key).
struct MapKey {
  const void* base;
  long long dim2;
  int dim1, d, box_rows, rank;
  bool bf16;
  bool operator==(const MapKey& o) const {
    return base == o.base && dim2 == o.dim2 && dim1 == o.dim1 && d == o.d && box_rows == o.box_rows &&
           rank == o.rank && bf16 == o.bf16;
  }
};
struct MapSlot {
  MapKey key;
  CUtensorMap map;
  bool valid;
};
constexpr int kMapCache = 64;
thread_local MapSlot t_maps[kMapCache];

MapSlot& map_slot(const MapKey& k) {
  uint64_t h = reinterpret_cast<uintptr_t>(k.base) * 0x9E3779B97F4A7C15ull;
  h ^= static_cast<uint64_t>(k.dim2) * 0xC2B2AE3D27D4EB4Full;
  h ^= (static_cast<uint64_t>(k.dim1) << 20) ^ (static_cast<uint64_t>(k.d) << 8) ^
       (static_cast<uint64_t>(k.box_rows) << 40) ^ (static_cast<uint64_t>(k.rank) << 56) ^ (k.bf16 ? 1u : 0u);
  h ^= h >> 29;
  return t_maps[h % kMapCache];
}

bool cached(CUtensorMap* m, const MapKey& k) {
  MapSlot& s = map_slot(k);
  if (!s.valid || !(s.key == k)) return false;
  *m = s.map;
  return true;
}

void remember(const CUtensorMap& m, const MapKey& k) {
  MapSlot& s = map_slot(k);
  s.key = k;
  s.map = m;
  s.valid = true;
}

// 3-D map over a [heads][N][d] row-major 16-bit tensor (heads = B*H); box = {64 elements, box_rows, 1};
// 128-byte swizzle. Rows past N are outside a head, so a tile that runs past the end of a sequence
// is zero-filled by the hardware instead of reading the next head's rows.
bool make_map(CUtensorMap* m, const void* base, long long heads, int N, int d, bool bf16, int box_rows) {
  const MapKey key{base, heads, N, d, box_rows, 3, bf16};
  if (cached(m, key)) return true;
  EncodeTiledFn enc = get_encode_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(heads)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2, static_cast<cuuint64_t>(N) * d * 2};
  cuuint32_t box[3] = {64u, static_cast<cuuint32_t>(box_rows), 1u};
  cuuint32_t estr[3] = {1u, 1u, 1u};
  CUresult r = enc(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
                   const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return false;
  remember(*m, key);
  return true;
}

// 2-D map over [rows][d] of a 16-bit tensor; box = {64 elements, box_rows}; 128-byte swizzle.
bool make_map_2d(CUtensorMap* m, const void* base, long long rows, int d, bool bf16, int box_rows) {
  const MapKey key{base, rows, 0, d, box_rows, 2, bf16};
  if (cached(m, key)) return true;
  EncodeTiledFn enc = get_encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(d) * 2};
  cuuint32_t box[2] = {64u, static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[2] = {1u, 1u};
  CUresult r = enc(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2,
                   const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return false;
  remember(*m, key);
  return true;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Paged decode shapes: d in {64, 128, 256}; page size a power of two in [16, 256]; the G = H / Hkv
// heads' Mq queries (G * Mq rows) fit one 128-row tile; cache rows and query rows in 32-bit ints.
fa_status check_decode_shape(int B, int H, int Hkv, int Mq, int d, int page_size, int n_pages, int max_pages,
                             fa_dtype dtype) {
  if (dtype != FA_F16 && dtype != FA_BF16) return FA_ERR_INVALID_ARG;
  if (B < 1 || H < 1 || Hkv < 1 || Mq < 1 || n_pages < 1 || max_pages < 1) return FA_ERR_UNSUPPORTED;
  if (d != 64 && d != 128 && d != 256) return FA_ERR_UNSUPPORTED;
  if (H % Hkv != 0 || (H / Hkv) * Mq > 128) return FA_ERR_UNSUPPORTED;
  if (page_size < 16 || page_size > 256 || (page_size & (page_size - 1)) != 0) return FA_ERR_UNSUPPORTED;
  if (static_cast<long long>(n_pages) * page_size >= (1ll << 31) ||
      static_cast<long long>(max_pages) * page_size >= (1ll << 31) ||
      static_cast<long long>(B) * H * Mq + 128 >= (1ll << 31))
    return FA_ERR_UNSUPPORTED;
  return FA_OK;
}

int log2_exact(int x) {
  int l = 0;
  while ((1 << l) < x) ++l;
  return l;
}

// Keys per decode tile (the kernel's BK) and the most splits the merge takes (its block is
// splits x d / 8 threads, at most 1024).
int decode_tile_keys(int d) { return d == 256 ? 64 : 128; }
int decode_max_splits(int d) { return d == 256 ? 32 : 64; }

// Splits of the key range: with C = B * Hkv CTAs per split and 152 SMs, pick the count s that
// minimises waves(C * s) * (tiles per split + 5), the 5 standing for a CTA's fixed cost in tiles
// (fitted to GB300 timings of split counts 1-24 on six decode shapes).
int decode_splits(int B, int Hkv, int d, int page_size, int max_pages) {
  const int bk = decode_tile_keys(d);
  const long long n_tiles = (static_cast<long long>(max_pages) * page_size + bk - 1) / bk;
  const long long ctas = static_cast<long long>(B) * Hkv;
  int best = 1;
  long long best_cost = -1;
  for (int s = 1; s <= decode_max_splits(d) && s <= n_tiles; ++s) {
    const long long waves = (ctas * s + 151) / 152;
    const long long cost = waves * ((n_tiles + s - 1) / s + 5);
    if (best_cost < 0 || cost < best_cost) {
      best_cost = cost;
      best = s;
    }
  }
  return best;
}

struct DecWs {
  size_t off_o, off_lse, total;
};
DecWs decode_ws(int B, int H, int Mq, int d, int n_split) {
  const size_t rows = static_cast<size_t>(B) * H * Mq, parts = static_cast<size_t>(n_split);
  DecWs w;
  w.off_o = 0;
  w.off_lse = (parts * rows * d * 4 + 255) & ~size_t(255);
  w.total = w.off_lse + ((parts * rows * 4 + 255) & ~size_t(255));
  return w;
}

fa_status check_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_CUDA;
  // 0 unknown, 1 a compute capability 10.3 device, 2 another device (the answer never changes)
  static std::atomic<unsigned char> known[64];
  if (dev >= 0 && dev < 64) {
    const unsigned char k = known[dev].load(std::memory_order_relaxed);
    if (k == 1) return FA_OK;
    if (k == 2) return FA_ERR_UNSUPPORTED;
  }
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess) return FA_ERR_CUDA;
  if (cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) return FA_ERR_CUDA;
  const bool ok = major == 10 && minor == 3;
  if (dev >= 0 && dev < 64) known[dev].store(ok ? 1 : 2, std::memory_order_relaxed);
  return ok ? FA_OK : FA_ERR_UNSUPPORTED;
}

constexpr int kMaxKeyBlocks = 65535;
constexpr int kMaxKvSplits = 16;

// Split-key forward: partial outputs [S][B*H*N][d] fp32 and their LSEs [S][B*H*N], each 256-byte aligned.
struct FwdWs {
  size_t off_o, off_lse, total;
};
FwdWs fwd_ws(int B, int H, int N, int d, int S) {
  const size_t rows = static_cast<size_t>(B) * H * N * S;
  FwdWs w;
  w.off_o = 0;
  w.off_lse = (rows * d * 4 + 255) & ~size_t(255);
  w.total = w.off_lse + ((rows * 4 + 255) & ~size_t(255));
  return w;
}

// The library's split count, from a cost model of the forward fitted to GB300 timings. A plain launch
// takes about max(longest item, total work / SMs) in (128-query x 128-key) tile pairs times the time a
// pair takes on one SM, plus a fixed cost for every wave of CTAs. A split shortens the longest item (the
// critical path under a causal mask or with few heads) but writes and re-reads an fp32 partial O per
// range and adds the merge launch. The count with the least modelled time wins; with many heads or
// short sequences that is 1.
int sm_count() {
  static std::atomic<int> cached{0};
  int n = cached.load(std::memory_order_relaxed);
  if (n > 0) return n;
  int dev = 0;
  n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) !=
                                                 cudaSuccess || n <= 0) {
    cudaGetLastError();
    n = 152;  // GB300
  }
  cached.store(n, std::memory_order_relaxed);
  return n;
}

double fwd_model_us(int B, int H, int N, int d, bool causal, int s, int sms) {
  const int NT = d <= 128 ? 2 : 1;
  const long long nq = (N + 127) / 128, nk = nq;
  const long long nblk = (nq + NT - 1) / NT;
  // the longest item is the last query block (causal) or any block (full); its first key range is full
  long long full = 0, longest = 0;
  const long long qt0 = (nblk - 1) * NT;
  for (long long t = qt0; t < qt0 + NT && t < nq; ++t) full = std::max(full, causal ? std::min(t + 1, nk) : nk);
  const long long per = (full + s - 1) / s;
  for (long long t = qt0; t < qt0 + NT && t < nq; ++t)
    longest += std::min(per, causal ? std::min(t + 1, nk) : nk);
  const double heads = static_cast<double>(B) * H;
  const double pairs = heads * (causal ? nk * (nk + 1) / 2.0 : static_cast<double>(nq) * nk);
  const double ctas = heads * nblk * s;
  const double t_pair = d == 64 ? 0.68 : d == 128 ? 0.75 : 2.4;  // us per tile pair on one SM
  double t = std::max(static_cast<double>(longest), 1.1 * pairs / sms) * t_pair + 1.5 * std::ceil(ctas / sms);
  if (s > 1) t += 4.0 + s * heads * N * d * 8.0 / 5.0e6;  // partials written and read at ~5 TB/s
  return t;
}

// Query tiles per work item of the forward without a split (d = 64, 128; 0 = the kernel's two, 1 = one).
// One tile an item doubles the items and halves the longest one, at the price of the tensor core
// waiting while the one softmax warpgroup works (with two tiles the two warpgroups keep it busy in
// turns): a step of one tile measured ~0.9 of a step of two. The choice is the smaller modelled
// makespan of the items, longest first on the SMs (each item: its key tiles times its step time plus a
// fixed cost of ~2 steps); it picked the faster mode on all 32 shapes measured (B2 H12, B1 H4, B4 H32;
// N = 512-4096; d = 64, 128; both masks). With more than four waves of one-tile items, two it is.
int fwd_tiles_per_item(int B, int H, int N, int d, bool causal) {
  if (d > 128) return 0;  // the d = 256 kernel takes one tile an item anyway
  const long long heads = static_cast<long long>(B) * H;
  const int nq = (N + 127) / 128;
  const int sms = sm_count();
  if (heads * nq > 4ll * sms) return 0;
  auto makespan = [&](int tpi) -> double {
    std::priority_queue<double, std::vector<double>, std::greater<double>> sm;
    for (int i = 0; i < sms; ++i) sm.push(0.0);
    // item classes longest first: under causal masking the last query tiles (or pairs) are the longest
    const int n_items = tpi == 1 ? nq : (nq + 1) / 2;
    for (int c = n_items - 1; c >= 0; --c) {
      const int steps = tpi == 1 ? (causal ? c + 1 : nq) : (causal ? std::min(2 * c + 2, nq) : nq);
      const double size = (tpi == 1 ? 0.9 : 1.0) * steps + 2.0;
      for (long long h = 0; h < heads; ++h) {
        const double t = sm.top();
        sm.pop();
        sm.push(t + size);
      }
    }
    double end = 0.0;
    while (!sm.empty()) {
      end = std::max(end, sm.top());
      sm.pop();
    }
    return end;
  };
  return makespan(1) < makespan(2) ? 1 : 0;
}

int fwd_kv_splits(int B, int H, int N, int d, bool causal) {
  const int sms = sm_count();
  const long long key_tiles = (N + 127) / 128;
  int best = 1;
  double best_t = fwd_model_us(B, H, N, d, causal, 1, sms);
  for (int s = 2; s <= kMaxKvSplits && s <= key_tiles; s *= 2) {
    const double t = fwd_model_us(B, H, N, d, causal, s, sms);
    if (t < best_t) best = s, best_t = t;
  }
  return best;
}

fa_status check_shape(int B, int H, int N, int d, fa_dtype dtype) {
  if (dtype != FA_F16 && dtype != FA_BF16) return FA_ERR_INVALID_ARG;
  if (B < 1 || H < 1 || N < 1) return FA_ERR_UNSUPPORTED;
  if (d != 64 && d != 128 && d != 256) return FA_ERR_UNSUPPORTED;
  // row indices (including the backward workspace's per-head padding) stay in 32-bit ints
  if (static_cast<long long>(B) * H * ((N + 127) / 128 * 128) >= (1ll << 31)) return FA_ERR_UNSUPPORTED;
  // the backward launches its 128-key blocks along the grid's y dimension (at most 65535)
  if ((N + 127) / 128 > kMaxKeyBlocks) return FA_ERR_UNSUPPORTED;
  return FA_OK;
}

fa_status check_scale(float scale) {
  if (!std::isfinite(scale) || !(scale > 0.f)) return FA_ERR_INVALID_ARG;
  return FA_OK;
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

struct WsLayout {
  size_t off_D, off_lse2, off_dq, total;
};
// Each head's rows are padded to Npad = N rounded up to 128: every 64-query step of the main
// kernel and every 128-row query tile of the separate dQ pass then starts 256-byte aligned (bulk
// copies need 16) and stays in its head; the last, partial step or tile of a sequence reads
// LSE*log2e and D of its own (zeroed, masked) padding rows and adds zero dQ partials there.
int pad_rows(int N) { return (N + 127) / 128 * 128; }
WsLayout ws_layout(int B, int H, int N, int d) {
  const size_t rows = static_cast<size_t>(B) * H * pad_rows(N);
  WsLayout w;
  w.off_D = 0;
  w.off_lse2 = align256(rows * 4);
  w.off_dq = w.off_lse2 + align256(rows * 4);
  w.total = w.off_dq + align256(rows * static_cast<size_t>(d) * 4);
  return w;
}

// Options resolved against the shape: K/V heads (0 = H, must divide H), key counts, fp32 O, how dQ
// is computed.
struct Opts {
  int Hkv;
  const int* kv_len;
  bool o_f32;
  int dq_mode;  // FA_DQ_DEFAULT, FA_DQ_ACCUMULATE or FA_DQ_SEPARATE
};
fa_status resolve_opts(const fa_options* opt, int H, const void* o_lo, Opts* out) {
  out->Hkv = H;
  out->kv_len = nullptr;
  out->o_f32 = false;
  out->dq_mode = FA_DQ_DEFAULT;
  if (!opt) return FA_OK;
  if (opt->dq_mode < FA_DQ_DEFAULT || opt->dq_mode > FA_DQ_SEPARATE) return FA_ERR_INVALID_ARG;
  out->dq_mode = opt->dq_mode;
  if (opt->n_kv_heads < 0) return FA_ERR_INVALID_ARG;
  if (opt->n_kv_heads > 0) {
    if (H % opt->n_kv_heads != 0) return FA_ERR_UNSUPPORTED;
    out->Hkv = opt->n_kv_heads;
  }
  if (opt->kv_len && (reinterpret_cast<uintptr_t>(opt->kv_len) & 3u) != 0) return FA_ERR_ALIGNMENT;
  out->kv_len = opt->kv_len;
  out->o_f32 = opt->o_fp32 != 0;
  if (out->o_f32 && o_lo) return FA_ERR_INVALID_ARG;  // the residual belongs to a 16-bit O
  return FA_OK;
}

// Whether dQ comes from the separate query-major pass: asked for explicitly (d = 64 or 128 only), or
// the library's choice, which follows the measured speed of the two paths per (d, mask).
fa_status dq_pass_for(const Opts& op, int d, bool causal, bool* out) {
  if (op.dq_mode == FA_DQ_SEPARATE) {
    if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
    *out = true;
    return FA_OK;
  }
  if (op.dq_mode == FA_DQ_ACCUMULATE || d == 256) {
    *out = false;
    return FA_OK;
  }
  (void)causal;
  *out = false;
  return FA_OK;
}

fa_status bwd_common(fa::BwdArgs* a, void* workspace, size_t workspace_bytes, int B, int H, int N, int d,
                     float scale, int causal, fa_dtype dtype, void* stream) {
  fa_status s = check_shape(B, H, N, d, dtype);
  if (s != FA_OK) return s;
  if ((s = check_scale(scale)) != FA_OK) return s;
  if (!workspace) return FA_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return FA_ERR_ALIGNMENT;
  WsLayout w = ws_layout(B, H, N, d);
  if (workspace_bytes < w.total) return FA_ERR_WORKSPACE;
  a->ws_D = reinterpret_cast<float*>(static_cast<char*>(workspace) + w.off_D);
  a->ws_lse2 = reinterpret_cast<float*>(static_cast<char*>(workspace) + w.off_lse2);
  a->ws_dqacc = reinterpret_cast<float*>(static_cast<char*>(workspace) + w.off_dq);
  a->B = B;
  a->H = H;
  a->Hkv = H;
  a->N = N;
  a->Npad = pad_rows(N);
  a->d = d;
  a->scale = scale;
  a->causal = causal != 0;
  a->bf16 = dtype == FA_BF16;
  a->timeout_ns = g_timeout_ns;
  a->stream = static_cast<cudaStream_t>(stream);
  return FA_OK;
}

fa_status bwd_preprocess_impl(const void* o, const void* o_lo, const void* dO, const float* lse, void* workspace,
                              size_t workspace_bytes, int B, int H, int N, int d, int causal, fa_dtype dtype,
                              const Opts& op, void* stream) {
  if (!o || !dO || !lse) return FA_ERR_INVALID_ARG;
  fa::BwdArgs a{};
  fa_status s = bwd_common(&a, workspace, workspace_bytes, B, H, N, d, 1.0f, 0, dtype, stream);
  if (s != FA_OK) return s;
  if (!aligned16(o) || !aligned16(o_lo) || !aligned16(dO) || !aligned16(lse)) return FA_ERR_ALIGNMENT;
  if ((s = check_device()) != FA_OK) return s;
  if ((s = dq_pass_for(op, d, causal, &a.dq_pass)) != FA_OK) return s;
  a.o = o;
  a.o_lo = o_lo;
  a.o_f32 = op.o_f32;
  a.dO = dO;
  a.lse = lse;
  return fa::launch_bwd_preprocess(a) == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

fa_status bwd_main_impl(const void* q, const void* k, const void* v, const void* dO, void* dk, void* dv, void* dq,
                        void* workspace, size_t workspace_bytes, int B, int H, int N, int d, float scale, int causal,
                        fa_dtype dtype, const Opts& op, void* stream) {
  if (!q || !k || !v || !dO || !dk || !dv) return FA_ERR_INVALID_ARG;
  fa::BwdArgs a{};
  fa_status s = bwd_common(&a, workspace, workspace_bytes, B, H, N, d, scale, causal, dtype, stream);
  if (s != FA_OK) return s;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(dO) || !aligned16(dk) || !aligned16(dv) ||
      !aligned16(dq))
    return FA_ERR_ALIGNMENT;
  if ((s = check_device()) != FA_OK) return s;
  if ((s = dq_pass_for(op, d, causal != 0, &a.dq_pass)) != FA_OK) return s;
  const int bq = fa::bwd_query_tile(d);
  if (bq == 0) return FA_ERR_UNSUPPORTED;
  const long long heads = static_cast<long long>(B) * H, kv_heads = static_cast<long long>(B) * op.Hkv;
  if (!make_map(&a.tm_q, q, heads, N, d, a.bf16, bq) || !make_map(&a.tm_do, dO, heads, N, d, a.bf16, bq) ||
      !make_map(&a.tm_k, k, kv_heads, N, d, a.bf16, 128) || !make_map(&a.tm_v, v, kv_heads, N, d, a.bf16, 128) ||
      !make_map(&a.tm_dk, dk, kv_heads, N, d, a.bf16, 128) || !make_map(&a.tm_dv, dv, kv_heads, N, d, a.bf16, 128))
    return FA_ERR_CUDA;
  a.Hkv = op.Hkv;
  a.kv_len = op.kv_len;
  a.dO = dO;
  a.dk = dk;
  a.dv = dv;
  a.dq = dq;  // optional: when given, the dQ conversion (or the dQ pass) is enqueued right after the main kernel
  return fa::launch_bwd_main(a) == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

fa_status bwd_dq_pass_impl(const void* q, const void* k, const void* v, const void* dO, void* dq, void* workspace,
                           size_t workspace_bytes, int B, int H, int N, int d, float scale, int causal, fa_dtype dtype,
                           const Opts& op, void* stream) {
  if (!q || !k || !v || !dO || !dq) return FA_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  fa::BwdArgs a{};
  fa_status s = bwd_common(&a, workspace, workspace_bytes, B, H, N, d, scale, causal, dtype, stream);
  if (s != FA_OK) return s;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(dO) || !aligned16(dq)) return FA_ERR_ALIGNMENT;
  if ((s = check_device()) != FA_OK) return s;
  const long long heads = static_cast<long long>(B) * H, kv_heads = static_cast<long long>(B) * op.Hkv;
  const int bq = fa::bwd_query_tile(d);
  if (!make_map(&a.tm_q, q, heads, N, d, a.bf16, bq) || !make_map(&a.tm_do, dO, heads, N, d, a.bf16, bq) ||
      !make_map(&a.tm_k, k, kv_heads, N, d, a.bf16, 128) || !make_map(&a.tm_v, v, kv_heads, N, d, a.bf16, 128))
    return FA_ERR_CUDA;
  a.Hkv = op.Hkv;
  a.kv_len = op.kv_len;
  a.dq_pass = true;
  a.dq = dq;
  return fa::launch_bwd_dq_pass(a) == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

}  // namespace

extern "C" {

int fa_version(void) { return 102; }

void fa_set_wait_timeout_ns(unsigned long long ns) { g_timeout_ns = ns ? ns : 4000000000ull; }

const char* fa_status_string(fa_status s) {
  switch (s) {
    case FA_OK: return "FA_OK";
    case FA_ERR_INVALID_ARG: return "FA_ERR_INVALID_ARG";
    case FA_ERR_UNSUPPORTED: return "FA_ERR_UNSUPPORTED";
    case FA_ERR_ALIGNMENT: return "FA_ERR_ALIGNMENT";
    case FA_ERR_WORKSPACE: return "FA_ERR_WORKSPACE";
    case FA_ERR_CUDA: return "FA_ERR_CUDA";
    case FA_ERR_TIMEOUT: return "FA_ERR_TIMEOUT";
    case FA_ERR_DEVICE_FAULT: return "FA_ERR_DEVICE_FAULT";
  }
  return "FA_ERR_UNKNOWN";
}

fa_status fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int d,
                 float scale, int causal, fa_dtype dtype, void* stream) {
  return fa_fwd_ex(q, k, v, o, lse, nullptr, B, H, N, d, scale, causal, dtype, stream);
}

fa_status fa_fwd_ex(const void* q, const void* k, const void* v, void* o, float* lse, void* o_lo, int B, int H, int N,
                    int d, float scale, int causal, fa_dtype dtype, void* stream) {
  return fa_fwd_opt(q, k, v, o, lse, o_lo, B, H, N, d, scale, causal, dtype, nullptr, stream);
}

fa_status fa_fwd_opt(const void* q, const void* k, const void* v, void* o, float* lse, void* o_lo, int B, int H,
                     int N, int d, float scale, int causal, fa_dtype dtype, const fa_options* opt, void* stream) {
  return fa_fwd_split(q, k, v, o, lse, o_lo, B, H, N, d, scale, causal, dtype, opt, 1, nullptr, 0, stream);
}

int fa_fwd_tiles_per_item(int B, int H, int N, int d, int causal) {
  if (check_shape(B, H, N, d, FA_BF16) != FA_OK) return 0;
  if (d > 128) return 1;
  return fwd_tiles_per_item(B, H, N, d, causal != 0) == 1 ? 1 : 2;
}

int fa_fwd_kv_splits(int B, int H, int N, int d, int causal) {
  if (check_shape(B, H, N, d, FA_BF16) != FA_OK) return 0;
  return fwd_kv_splits(B, H, N, d, causal != 0);
}

size_t fa_fwd_workspace_size(int B, int H, int N, int d, int kv_splits) {
  if (check_shape(B, H, N, d, FA_BF16) != FA_OK || kv_splits < 2 || kv_splits > kMaxKvSplits) return 0;
  return fwd_ws(B, H, N, d, kv_splits).total;
}

fa_status fa_fwd_split(const void* q, const void* k, const void* v, void* o, float* lse, void* o_lo, int B, int H,
                       int N, int d, float scale, int causal, fa_dtype dtype, const fa_options* opt, int kv_splits,
                       void* workspace, size_t workspace_bytes, void* stream) {
  if (!q || !k || !v || !o || !lse) return FA_ERR_INVALID_ARG;
  fa_status s = check_shape(B, H, N, d, dtype);
  if (s != FA_OK) return s;
  if ((s = check_scale(scale)) != FA_OK) return s;
  Opts op;
  if ((s = resolve_opts(opt, H, o_lo, &op)) != FA_OK) return s;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse) || !aligned16(o_lo))
    return FA_ERR_ALIGNMENT;
  if ((s = check_device()) != FA_OK) return s;
  fa::FwdArgs a;
  const bool bf16 = dtype == FA_BF16;
  const long long heads = static_cast<long long>(B) * H, kv_heads = static_cast<long long>(B) * op.Hkv;
  if (!make_map(&a.tm_q, q, heads, N, d, bf16, 128) || !make_map(&a.tm_k, k, kv_heads, N, d, bf16, 128) ||
      !make_map(&a.tm_v, v, kv_heads, N, d, bf16, 128))
    return FA_ERR_CUDA;
  if (kv_splits <= 0) kv_splits = fwd_kv_splits(B, H, N, d, causal != 0);
  if (kv_splits > kMaxKvSplits) return FA_ERR_UNSUPPORTED;
  a.kv_splits = kv_splits;
  a.tiles_per_item = kv_splits > 1 ? 0 : fwd_tiles_per_item(B, H, N, d, causal != 0);
  a.part_o = nullptr;
  a.part_lse = nullptr;
  if (kv_splits > 1) {
    const FwdWs w = fwd_ws(B, H, N, d, kv_splits);
    if (!workspace) return FA_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return FA_ERR_ALIGNMENT;
    if (workspace_bytes < w.total) return FA_ERR_WORKSPACE;
    a.part_o = reinterpret_cast<float*>(static_cast<char*>(workspace) + w.off_o);
    a.part_lse = reinterpret_cast<float*>(static_cast<char*>(workspace) + w.off_lse);
  }
  a.o = o;
  a.lse = lse;
  a.o_lo = o_lo;
  a.kv_len = op.kv_len;
  a.B = B;
  a.H = H;
  a.Hkv = op.Hkv;
  a.N = N;
  a.d = d;
  a.o_f32 = op.o_f32;
  a.scale = scale;
  a.causal = causal != 0;
  a.bf16 = bf16;
  a.timeout_ns = g_timeout_ns;
  a.stream = static_cast<cudaStream_t>(stream);
  return fa::launch_fwd(a) == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

size_t fa_bwd_workspace_size(int B, int H, int N, int d) {
  if (check_shape(B, H, N, d, FA_BF16) != FA_OK) return 0;
  return ws_layout(B, H, N, d).total;
}

fa_status fa_bwd_preprocess(const void* o, const void* o_lo, const void* dO, const float* lse, void* workspace,
                            size_t workspace_bytes, int B, int H, int N, int d, fa_dtype dtype, void* stream) {
  return bwd_preprocess_impl(o, o_lo, dO, lse, workspace, workspace_bytes, B, H, N, d, 0, dtype,
                             Opts{H, nullptr, false, FA_DQ_ACCUMULATE}, stream);
}

fa_status fa_bwd_preprocess_opt(const void* o, const void* o_lo, const void* dO, const float* lse, void* workspace,
                                size_t workspace_bytes, int B, int H, int N, int d, int causal, fa_dtype dtype,
                                const fa_options* opt, void* stream) {
  Opts op;
  fa_status s = resolve_opts(opt, H, o_lo, &op);
  if (s != FA_OK) return s;
  return bwd_preprocess_impl(o, o_lo, dO, lse, workspace, workspace_bytes, B, H, N, d, causal, dtype, op, stream);
}

fa_status fa_bwd_main(const void* q, const void* k, const void* v, const void* dO, void* dk, void* dv, void* dq,
                      void* workspace, size_t workspace_bytes, int B, int H, int N, int d, float scale, int causal,
                      fa_dtype dtype, void* stream) {
  return bwd_main_impl(q, k, v, dO, dk, dv, dq, workspace, workspace_bytes, B, H, N, d, scale, causal, dtype,
                       Opts{H, nullptr, false, FA_DQ_ACCUMULATE}, stream);
}

fa_status fa_bwd_main_opt(const void* q, const void* k, const void* v, const void* dO, void* dk, void* dv, void* dq,
                          void* workspace, size_t workspace_bytes, int B, int H, int N, int d, float scale, int causal,
                          fa_dtype dtype, const fa_options* opt, void* stream) {
  Opts op;
  fa_status s = resolve_opts(opt, H, nullptr, &op);
  if (s != FA_OK) return s;
  return bwd_main_impl(q, k, v, dO, dk, dv, dq, workspace, workspace_bytes, B, H, N, d, scale, causal, dtype, op,
                       stream);
}

int fa_bwd_uses_dq_pass(int d, int causal, const fa_options* opt) {
  Opts op{1, nullptr, false, opt ? opt->dq_mode : FA_DQ_DEFAULT};
  if (op.dq_mode < FA_DQ_DEFAULT || op.dq_mode > FA_DQ_SEPARATE) return 0;
  bool pass = false;
  if (dq_pass_for(op, d, causal != 0, &pass) != FA_OK) return 0;
  return pass ? 1 : 0;
}

fa_status fa_bwd_dq_pass(const void* q, const void* k, const void* v, const void* dO, void* dq, void* workspace,
                         size_t workspace_bytes, int B, int H, int N, int d, float scale, int causal, fa_dtype dtype,
                         const fa_options* opt, void* stream) {
  Opts op;
  fa_status s = resolve_opts(opt, H, nullptr, &op);
  if (s != FA_OK) return s;
  return bwd_dq_pass_impl(q, k, v, dO, dq, workspace, workspace_bytes, B, H, N, d, scale, causal, dtype, op, stream);
}

fa_status fa_bwd_dq_convert(void* dq, const void* workspace, size_t workspace_bytes, int B, int H, int N, int d,
                            float scale, fa_dtype dtype, void* stream) {
  if (!dq) return FA_ERR_INVALID_ARG;
  fa::BwdArgs a{};
  fa_status s = bwd_common(&a, const_cast<void*>(workspace), workspace_bytes, B, H, N, d, scale, 0, dtype, stream);
  if (s != FA_OK) return s;
  if (!aligned16(dq)) return FA_ERR_ALIGNMENT;
  if ((s = check_device()) != FA_OK) return s;
  a.dq = dq;
  return fa::launch_bwd_dq_convert(a) == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

fa_status fa_bwd(const void* q, const void* k, const void* v, const void* o, const void* dO, const float* lse,
                 void* dq, void* dk, void* dv, const void* o_lo, void* workspace, size_t workspace_bytes, int B, int H,
                 int N, int d, float scale, int causal, fa_dtype dtype, void* stream) {
  return fa_bwd_opt(q, k, v, o, dO, lse, dq, dk, dv, o_lo, workspace, workspace_bytes, B, H, N, d, scale, causal,
                    dtype, nullptr, stream);
}

fa_status fa_bwd_opt(const void* q, const void* k, const void* v, const void* o, const void* dO, const float* lse,
                     void* dq, void* dk, void* dv, const void* o_lo, void* workspace, size_t workspace_bytes, int B,
                     int H, int N, int d, float scale, int causal, fa_dtype dtype, const fa_options* opt,
                     void* stream) {
  if (!q || !k || !v || !o || !dO || !lse || !dq || !dk || !dv) return FA_ERR_INVALID_ARG;
  // Validate everything before enqueuing anything.
  fa::BwdArgs probe{};
  fa_status s = bwd_common(&probe, workspace, workspace_bytes, B, H, N, d, scale, causal, dtype, stream);
  if (s != FA_OK) return s;
  Opts op;
  if ((s = resolve_opts(opt, H, o_lo, &op)) != FA_OK) return s;
  if (fa::bwd_query_tile(d) == 0) return FA_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(dO) || !aligned16(lse) ||
      !aligned16(dq) || !aligned16(dk) || !aligned16(dv) || !aligned16(o_lo))
    return FA_ERR_ALIGNMENT;
  if ((s = check_device()) != FA_OK) return s;
  bool dq_pass = false;
  if ((s = dq_pass_for(op, d, causal != 0, &dq_pass)) != FA_OK) return s;
  if ((s = bwd_preprocess_impl(o, o_lo, dO, lse, workspace, workspace_bytes, B, H, N, d, causal, dtype, op, stream)) !=
      FA_OK)
    return s;
  // given dq, the main kernel's launch enqueues the dQ conversion right after it
  return bwd_main_impl(q, k, v, dO, dk, dv, dq, workspace, workspace_bytes, B, H, N, d, scale, causal, dtype, op,
                       stream);
}

int fa_decode_splits(int B, int Hkv, int d, int page_size, int max_pages) {
  if (B < 1 || Hkv < 1 || page_size < 1 || max_pages < 1 || (d != 64 && d != 128 && d != 256)) return 0;
  return decode_splits(B, Hkv, d, page_size, max_pages);
}

size_t fa_decode_workspace_size(int B, int H, int Hkv, int Mq, int d, int page_size, int max_pages, int n_split) {
  if (check_decode_shape(B, H, Hkv, Mq, d, page_size, 1, max_pages, FA_BF16) != FA_OK) return 0;
  if (n_split <= 0) n_split = decode_splits(B, Hkv, d, page_size, max_pages);
  if (n_split > decode_max_splits(d)) n_split = decode_max_splits(d);
  return decode_ws(B, H, Mq, d, n_split).total;
}

fa_status fa_decode(const void* q, const void* k_pages, const void* v_pages, const int* page_table, const int* ctx_len,
                    void* o, float* lse, void* workspace, size_t workspace_bytes, int B, int H, int Hkv, int Mq, int d,
                    int page_size, int n_pages, int max_pages, int n_split, float scale, int causal, fa_dtype dtype,
                    void* stream) {
  if (!q || !k_pages || !v_pages || !page_table || !ctx_len || !o || !lse) return FA_ERR_INVALID_ARG;
  fa_status s = check_decode_shape(B, H, Hkv, Mq, d, page_size, n_pages, max_pages, dtype);
  if (s != FA_OK) return s;
  if ((s = check_scale(scale)) != FA_OK) return s;
  if (n_split <= 0) n_split = decode_splits(B, Hkv, d, page_size, max_pages);
  if (n_split > decode_max_splits(d)) n_split = decode_max_splits(d);
  const int bk = decode_tile_keys(d);
  const long long n_tiles = (static_cast<long long>(max_pages) * page_size + bk - 1) / bk;
  if (n_split > n_tiles) n_split = static_cast<int>(n_tiles);
  const int tiles_per_split = static_cast<int>((n_tiles + n_split - 1) / n_split);
  n_split = static_cast<int>((n_tiles + tiles_per_split - 1) / tiles_per_split);  // no empty trailing split
  const DecWs w = decode_ws(B, H, Mq, d, n_split);
  if (!workspace) return FA_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return FA_ERR_ALIGNMENT;
  if (workspace_bytes < w.total) return FA_ERR_WORKSPACE;
  if (!aligned16(q) || !aligned16(k_pages) || !aligned16(v_pages) || !aligned16(o) || !aligned16(lse) ||
      (reinterpret_cast<uintptr_t>(page_table) & 3u) != 0 || (reinterpret_cast<uintptr_t>(ctx_len) & 3u) != 0)
    return FA_ERR_ALIGNMENT;
  if ((s = check_device()) != FA_OK) return s;
  fa::DecArgs a;
  const bool bf16 = dtype == FA_BF16;
  const int br = page_size < bk ? page_size : bk;
  if (!make_map_2d(&a.tm_q, q, static_cast<long long>(B) * H * Mq, d, bf16, 128) ||
      !make_map(&a.tm_k, k_pages, Hkv, n_pages * page_size, d, bf16, br) ||
      !make_map(&a.tm_v, v_pages, Hkv, n_pages * page_size, d, bf16, br))
    return FA_ERR_CUDA;
  a.page_table = page_table;
  a.ctx_len = ctx_len;
  a.ws_o = reinterpret_cast<float*>(static_cast<char*>(workspace) + w.off_o);
  a.ws_lse = reinterpret_cast<float*>(static_cast<char*>(workspace) + w.off_lse);
  a.o = o;
  a.lse = lse;
  a.B = B;
  a.H = H;
  a.Hkv = Hkv;
  a.Mq = Mq;
  a.d = d;
  a.ps_log2 = log2_exact(page_size);
  a.max_pages = max_pages;
  a.n_pages = n_pages;
  a.tiles_per_split = tiles_per_split;
  a.n_split = n_split;
  a.scale = scale;
  a.causal = causal != 0;
  a.bf16 = bf16;
  a.timeout_ns = g_timeout_ns;
  a.stream = static_cast<cudaStream_t>(stream);
  return fa::launch_decode(a) == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

fa_status fa_device_status(void* stream, unsigned int info[4]) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(st) != cudaSuccess) return FA_ERR_CUDA;
  fa::DevStatusHost a{}, b{}, c{}, t{};
  if (fa::read_clear_status_fwd(&a, st) != cudaSuccess) return FA_ERR_CUDA;
  if (fa::read_clear_status_bwd(&b, st) != cudaSuccess) return FA_ERR_CUDA;
  if (fa::read_clear_status_decode(&c, st) != cudaSuccess) return FA_ERR_CUDA;
  if (fa::read_clear_status_selftest(&t, st) != cudaSuccess) return FA_ERR_CUDA;
  const fa::DevStatusHost& first = a.code ? a : (b.code ? b : (c.code ? c : t));
  if (info) {
    info[0] = first.code;
    info[1] = first.where;
    info[2] = first.block;
    info[3] = a.count + b.count + c.count + t.count;
  }
  if (first.code == 1u) return FA_ERR_TIMEOUT;
  if (first.code != 0u) return FA_ERR_DEVICE_FAULT;
  return FA_OK;
}

}  // extern "C"
