// Launch order of the backward main kernels' (K/V head, 128-key block) work items.
//
// One CTA is launched per item, and CTAs start (or, in the persistent kernels, are taken over)
// in the order of blockIdx.x + gridDim.x * blockIdx.y. The order takes the K/V heads in groups
// and, within a group, the key blocks in ascending order (block 0, the longest under causal
// masking, first) across the group's heads. The CTAs in flight then share the Q, dO and fp32 dQ
// rows of a few heads, which stay in L2, while long blocks still start before short ones.
#pragma once

namespace fa {

// Maps the launch index (x, y) of a grid of `heads` x `nkb` CTAs to the K/V head `bh` and key
// block `kb` it works on. head_bytes: the rows one K/V head's blocks share (G query heads x N rows
// x (2 + 2 + 4) bytes x d). Groups are kept to about 64 MB of such rows, and to no more than
// heads * nkb / 304 groups: a causal block 0 takes about 304 / (heads * nkb) of the run on 152
// SMs, and a group's block 0 starts only when that group does, so more groups would lengthen the
// run's tail. The map is a bijection for every heads, nkb >= 1.
__device__ __forceinline__ void bwd_block_order(int x, int y, int heads, int nkb, long long head_bytes, int& bh,
                                                int& kb) {
  const long long fit = (64ll << 20) / (head_bytes > 0 ? head_bytes : 1);
  const int hg_max = fit < 1 ? 1 : (fit > heads ? heads : static_cast<int>(fit));
  const int ng_mem = (heads + hg_max - 1) / hg_max;
  const long long ng_tail_ll = static_cast<long long>(heads) * nkb / 304;
  const int ng_tail = ng_tail_ll < 1 ? 1 : (ng_tail_ll > heads ? heads : static_cast<int>(ng_tail_ll));
  const int ng = ng_mem < ng_tail ? ng_mem : ng_tail;
  const int hg = (heads + ng - 1) / ng;  // heads per group
  const int lin = x + heads * y;
  const int gi = lin / (hg * nkb), r = lin - gi * hg * nkb;
  const int gh = heads - gi * hg < hg ? heads - gi * hg : hg;  // heads in this group (the last may have fewer)
  bh = gi * hg + r % gh;
  kb = r / gh;
}

}  // namespace fa
