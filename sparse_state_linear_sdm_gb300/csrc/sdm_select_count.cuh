// Counting selection of bf16 sub-scores (Sparse Delta Memory technical summary,
// gist.science/it/paper/2607.07386, "Meccanismo Core" item 2): the same results as the
// general selection in sdm_select_impl.cuh, bit for bit, with far fewer instructions for
// the inputs the layer sees.
//
// Inner top-k of a half.  Positive bf16 values are ordered like their 16-bit patterns.
// When the largest value of a half is positive (pattern `top`), the candidates for its
// top-k are the values whose pattern lies in [top - 255, top]: one histogram with one bin
// per pattern (bin = top - pattern; negative values and zeros fall outside) and its prefix
// sums give every selected value its place in the output, so the selection and the
// ordering are one scatter, with no radix passes and no sorting network.  The halves stay
// in registers after their 16-byte loads.  Values that share a pattern land in their
// bin's range in arbitrary order and each bin is then put in index order; at the cut, the
// values of the boundary bin (at most 32) are ranked against each other.
//
// Outer top-K over the staircase of pair sums (p+1)(q+1) <= K.  When every staircase sum
// is positive, the fp32 patterns of the sums are ordered like the sums, and 256 bins over
// [smallest row-end sum, largest sum] (a bin can hold several sums: each bin is sorted by
// the full key) place the candidates the same way.  The pass that guards against fp32
// rounding merges (pairs beyond the staircase that could beat the K-th key) is skipped
// when all pair sums are exact: bf16 values whose exponents span at most 15 add exactly
// in fp32 (8 + 15 + 1 significant bits).
//
// Whenever a precondition does not hold (a half whose largest value is not a positive
// normal number, fewer than k values in the window, more than 32 at the cut; sums that
// are not all positive, a window narrower than 256 sum patterns), that half or that outer
// selection takes the general path's radix select and sort on the same keys, so every
// input is handled exactly.
//
// One warp per (b, h, t, k'-or-q') task, as in the general path.  The inner lists are
// kept packed: bf16 pattern << 16 | index in one 32-bit word.
#pragma once

#include "sdm_select_impl.cuh"

namespace sdm {
namespace {

constexpr int kCountMaxS = 1024;  // four 16-byte loads per lane and half
constexpr int kCountMaxK = 128;   // four output slots per lane
constexpr int kBoundMax = 32;     // keys sharing the cut's bin, ranked one per lane
constexpr int kGroupMax = 96;     // bins before the cut holding two keys or more

// One warp's shared memory: keys (the general path's keys, or the outer candidates), the
// selected outer keys, 256 bins (count << 16 | cursor) and one junk bin per lane, the two
// packed inner lists, the boundary keys followed by one junk slot per lane, and the list of
// bins that need ordering.
constexpr int kBinWords = 256 + 32;
struct CountSmem {
  unsigned char* keys;
  unsigned char* out;
  uint32_t* bins;
  uint32_t* la;  // half 0's list: bf16 pattern << 16 | index
  uint32_t* lb;  // half 1's list
  unsigned char* tmp;
  uint32_t* groups;
};

__host__ __device__ inline size_t count_lists_bytes(int kin_max) {
  return (size_t(2) * kin_max * 4 + 15) / 16 * 16;
}
__host__ __device__ inline size_t count_per_warp_bytes(size_t keys_bytes, int kpad, int kin_max) {
  return keys_bytes + size_t(kpad) * 8 + kBinWords * 4 + count_lists_bytes(kin_max) +
         2 * kBoundMax * 8 + kGroupMax * 4;
}

__device__ __forceinline__ CountSmem count_smem(unsigned char* wp, size_t keys_bytes, int kpad,
                                                int kin_max) {
  CountSmem m;
  m.keys = wp;
  m.out = wp + keys_bytes;
  m.bins = reinterpret_cast<uint32_t*>(m.out + size_t(kpad) * 8);
  m.la = m.bins + kBinWords;
  m.lb = m.la + kin_max;
  m.tmp = reinterpret_cast<unsigned char*>(m.bins + kBinWords) + count_lists_bytes(kin_max);
  m.groups = reinterpret_cast<uint32_t*>(m.tmp + 2 * kBoundMax * 8);
  return m;
}

__device__ __forceinline__ uint32_t saddr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Packed list entry of a general-path inner key (value pattern << 16 | index).
__device__ __forceinline__ uint32_t pack_inner(uint32_t key) {
  const uint32_t o = key >> 16;
  const uint32_t b = (o & 0x8000u) ? (o & 0x7FFFu) : (~o & 0xFFFFu);
  return (b << 16) | (0xFFFFu - (key & 0xFFFFu));
}
__device__ __forceinline__ float entry_value(uint32_t e) { return __uint_as_float(e & 0xFFFF0000u); }
__device__ __forceinline__ uint32_t entry_index(uint32_t e) { return e & 0xFFFFu; }

// bins[bin] += 1 << 16 (the count half of the bin word) when bin < 256, else the lane's junk
// bin: no branch.
__device__ __forceinline__ void bin_count(uint32_t* bins, uint32_t bin, uint32_t junk) {
  atomicAdd(&bins[min(bin, junk)], 0x10000u);
}

// Places an entry of bin `bin`: when bin <= bstar it takes the bin's cursor (low half of the
// bin word, post-incremented) as its position, in dst (bin < bstar) or in tmp (bin == bstar);
// otherwise it goes to the lane's junk slot.  No branch.
template <typename Key>
__device__ __forceinline__ void bin_place(uint32_t* bins, uint32_t bin, uint32_t bstar,
                                          uint32_t junk, Key* dst, Key* tmp, Key* jslot, Key e) {
  const bool le = bin <= bstar;
  const uint32_t pos = atomicAdd(&bins[le ? bin : junk], le ? 1u : 0u) & 0xFFFFu;
  Key* base = bin < bstar ? dst : (le ? tmp : jslot);
  base[le ? pos : 0u] = e;
}

// The bins hold key counts in their high 16 bits, bin 0 for the largest keys; lane l owns
// bins 8l .. 8l+7.  Finds the bin holding the need-th largest key (bstar, with `above` keys
// in earlier bins and `cnt` in bstar itself), turns every bin into count << 16 | cursor, the
// cursor starting at the bin's first position (bins before bstar) or at 0 (bstar, whose keys
// go to the boundary buffer), and lists the bins before bstar that hold two keys or more as
// count << 16 | first position in groups[0..ngroups).  Returns false (warp-uniform) when
// the bins hold fewer than need keys, when more than kBoundMax keys share bstar, or when
// more than kGroupMax bins would need ordering.
__device__ __forceinline__ bool count_scan(uint32_t* bins, int need, uint32_t* groups,
                                           int& ngroups, int& bstar, uint32_t& above,
                                           uint32_t& cnt) {
  const int lane = threadIdx.x & 31;
  uint4* b4 = reinterpret_cast<uint4*>(bins);
  const uint4 v0 = b4[2 * lane], v1 = b4[2 * lane + 1];
  uint32_t c[8];
  c[0] = v0.x >> 16; c[1] = v0.y >> 16; c[2] = v0.z >> 16; c[3] = v0.w >> 16;
  c[4] = v1.x >> 16; c[5] = v1.y >> 16; c[6] = v1.z >> 16; c[7] = v1.w >> 16;
  uint32_t s = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) s += c[i];
  uint32_t incl = s;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const uint32_t y = __shfl_up_sync(kFull, incl, off);
    if (lane >= off) incl += y;
  }
  const uint32_t total = __shfl_sync(kFull, incl, 31);
  if (total < uint32_t(need)) return false;
  uint32_t run = incl - s, w[8], ab = 0, ct = 0;
  int d = -1;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const bool cut = run < uint32_t(need) && run + c[i] >= uint32_t(need);
    w[i] = (c[i] << 16) | (cut ? 0u : run);
    if (cut) {
      d = 8 * lane + i;
      ab = run;
      ct = c[i];
    }
    run += c[i];
  }
  b4[2 * lane] = make_uint4(w[0], w[1], w[2], w[3]);
  b4[2 * lane + 1] = make_uint4(w[4], w[5], w[6], w[7]);
  const int owner = __ffs(__ballot_sync(kFull, d >= 0)) - 1;
  bstar = __shfl_sync(kFull, d, owner);
  above = __shfl_sync(kFull, ab, owner);
  cnt = __shfl_sync(kFull, ct, owner);
  if (cnt > uint32_t(kBoundMax)) return false;
  // bins before the cut with two keys or more, listed in bin order
  uint32_t tie = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) tie |= (8 * lane + i < bstar && c[i] > 1u) ? (1u << i) : 0u;
  const uint32_t nt = __popc(tie);
  uint32_t tincl = nt;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const uint32_t y = __shfl_up_sync(kFull, tincl, off);
    if (lane >= off) tincl += y;
  }
  ngroups = int(__shfl_sync(kFull, tincl, 31));
  if (ngroups > kGroupMax) return false;
  uint32_t g = tincl - nt;
#pragma unroll
  for (int i = 0; i < 8; ++i)
    if (tie & (1u << i)) groups[g++] = (c[i] << 16) | (w[i] & 0xFFFFu);
  __syncwarp();
  return true;
}

// After the scatter: dst[0..above) holds the keys of the bins before the cut, each bin's
// keys in its range in arbitrary order; tmp[0..cnt) the keys of the cut's bin.  Ranks the cut's
// keys and places the first need = k - above after the others, then sorts each listed bin's
// range (one lane per bin) so that dst[0..k) is in order (`before(x, y)`: x comes first).
// Keys are distinct.
template <typename Key, class Before>
__device__ __forceinline__ void count_finish(Key* dst, const Key* tmp, const uint32_t* groups,
                                             int ngroups, int k, uint32_t above, uint32_t cnt,
                                             const Before& before) {
  const int lane = threadIdx.x & 31;
  const int need = k - int(above);
  const Key mine = lane < int(cnt) ? tmp[lane] : Key(0);
  int rank = 0;
  for (int j = 0; j < int(cnt); ++j) rank += before(__shfl_sync(kFull, mine, j), mine) ? 1 : 0;
  if (lane < int(cnt) && rank < need) dst[above + rank] = mine;
  for (int g = lane; g < ngroups; g += 32) {
    const uint32_t d = groups[g];
    const int s = int(d & 0xFFFFu), e = s + int(d >> 16);
    for (int a = s + 1; a < e; ++a) {
      const Key x = dst[a];
      int b = a - 1;
      while (b >= s && before(x, dst[b])) {
        dst[b + 1] = dst[b];
        --b;
      }
      dst[b + 1] = x;
    }
  }
  __syncwarp();
}

__device__ bool inner_count_raw(const uint4* raw, int S, int kin, int top, const CountSmem& m,
                                uint32_t* lst);

// Top-kin of one bf16 half (S values, 16-byte aligned, S % 8 == 0, S <= kCountMaxS) by
// (value desc, index asc), packed into lst[0..kin); the half's 16-byte chunks are kept in
// the keys region between passes.  Returns false when the half's largest
// value is not a positive number of pattern >= 256, when fewer than kin values lie within
// 256 patterns of it, or when more than kBoundMax share the value at the cut (lst is then
// unspecified and the caller takes the general path).
__device__ bool inner_count(const uint16_t* src, int S, int kin, const CountSmem& m,
                            uint32_t* lst) {
  const int lane = threadIdx.x & 31;
  const uint4* src4 = reinterpret_cast<const uint4*>(src);
  uint4* raw = reinterpret_cast<uint4*>(m.keys);  // the half's 16-byte chunks, as loaded
  const int nvec = S >> 3;
  constexpr int U = kCountMaxS / 256;
  // Chunk c = lane + 32u holds values 8c .. 8c+7.  All loads are issued before any is used.
  uint4 q[U];
#pragma unroll
  for (int u = 0; u < U; ++u) {
    const int c = lane + 32 * u;
    q[u] = c < nvec ? __ldg(src4 + c) : make_uint4(0x80008000u, 0x80008000u, 0x80008000u, 0x80008000u);
  }
  // 1. the largest pattern read as a signed 16-bit number (positive values: the largest value)
  uint32_t mx2 = 0x80008000u;
#pragma unroll
  for (int u = 0; u < U; ++u) {
    mx2 = __vmaxs2(__vmaxs2(mx2, q[u].x), __vmaxs2(q[u].y, __vmaxs2(q[u].z, q[u].w)));
    if (lane + 32 * u < nvec) raw[lane + 32 * u] = q[u];
  }
  const int mxl = max(int(int16_t(mx2 & 0xFFFFu)), int(int16_t(mx2 >> 16)));
  const int top = __reduce_max_sync(kFull, mxl);
  if (top < 256) return false;
  __syncwarp();
  return inner_count_raw(raw, S, kin, top, m, lst);
}

// inner_count on a half already in shared memory (16-byte aligned, S % 8 == 0, S <=
// kCountMaxS); the same result.
__device__ bool inner_count_smem(const uint16_t* half, int S, int kin, const CountSmem& m,
                                 uint32_t* lst) {
  const int lane = threadIdx.x & 31;
  const uint4* raw = reinterpret_cast<const uint4*>(half);
  uint32_t mx2 = 0x80008000u;
  for (int c = lane; c < (S >> 3); c += 32) {
    const uint4 q = raw[c];
    mx2 = __vmaxs2(__vmaxs2(mx2, q.x), __vmaxs2(q.y, __vmaxs2(q.z, q.w)));
  }
  const int mxl = max(int(int16_t(mx2 & 0xFFFFu)), int(int16_t(mx2 >> 16)));
  const int top = __reduce_max_sync(kFull, mxl);
  if (top < 256) return false;
  return inner_count_raw(raw, S, kin, top, m, lst);
}

// Steps 2-5 of inner_count on the half's 16-byte chunks `raw` (shared memory), whose largest
// pattern is top >= 256.
__device__ bool inner_count_raw(const uint4* raw, int S, int kin, int top, const CountSmem& m,
                                uint32_t* lst) {
  const int lane = threadIdx.x & 31;
  const int nvec = S >> 3;
  uint32_t* bins = m.bins;
  const uint32_t junk = 256u + uint32_t(lane);
  reinterpret_cast<uint4*>(bins)[2 * lane] = make_uint4(0u, 0u, 0u, 0u);
  reinterpret_cast<uint4*>(bins)[2 * lane + 1] = make_uint4(0u, 0u, 0u, 0u);
  __syncwarp();
  // 2. histogram of the patterns top - 255 .. top (bin = top - pattern)
#pragma unroll 1
  for (int c = lane; c < nvec; c += 32) {
    const uint4 x = raw[c];
    const uint32_t w4[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      bin_count(bins, uint32_t(top) - (w4[k] & 0xFFFFu), junk);
      bin_count(bins, uint32_t(top) - (w4[k] >> 16), junk);
    }
  }
  __syncwarp();
  // 3. the cut, the bins' cursors and the bins to order
  uint32_t above, cnt;
  int bstar, ngroups;
  if (!count_scan(bins, kin, m.groups, ngroups, bstar, above, cnt)) return false;
  // 4. scatter: entries pattern << 16 | index of the bins up to the cut
  uint32_t* tmp = reinterpret_cast<uint32_t*>(m.tmp);
  uint32_t* jslot = tmp + kBoundMax + lane;
#pragma unroll 1
  for (int c = lane; c < nvec; c += 32) {
    const uint4 x = raw[c];
    const uint32_t w4[4] = {x.x, x.y, x.z, x.w};
    const uint32_t j0 = uint32_t(8 * c);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      bin_place<uint32_t>(bins, uint32_t(top) - (w4[k] & 0xFFFFu), uint32_t(bstar), junk, lst, tmp,
                          jslot, (w4[k] << 16) | (j0 + 2 * k));
      bin_place<uint32_t>(bins, uint32_t(top) - (w4[k] >> 16), uint32_t(bstar), junk, lst, tmp,
                          jslot, (w4[k] & 0xFFFF0000u) | (j0 + 2 * k + 1));
    }
  }
  __syncwarp();
  // 5. the cut's values by index, every bin in index order (same pattern: entry order)
  count_finish<uint32_t>(lst, tmp, m.groups, ngroups, kin, above, cnt,
                         [](uint32_t x, uint32_t y) { return x < y; });
  return true;
}

// The general path for one bf16 half (radix select on the keys, then a bitonic sort),
// packed into lst.
__device__ __noinline__ void inner_general(const uint16_t* src, int S, int kin, bool vec, const CountSmem& m,
                              uint32_t* lst) {
  const int lane = threadIdx.x & 31;
  uint32_t* ik = reinterpret_cast<uint32_t*>(m.keys);
  uint32_t* io = reinterpret_cast<uint32_t*>(m.out);
  load_half_keys<uint16_t>(src, S, vec, ik, m.bins);
  warp_topk_from<uint32_t>(ik, S, kin, io, m.bins, 0u, InnerKeyOf<uint16_t>::top_shift, true, 16);
  sort_desc_upto<uint32_t, 4>(io, kin);
  for (int r = lane; r < kin; r += 32) lst[r] = pack_inner(io[r]);
  __syncwarp();
}

// inner_general on a half already in shared memory.
__device__ __noinline__ void inner_general_smem(const uint16_t* half, int S, int kin,
                                                const CountSmem& m, uint32_t* lst) {
  const int lane = threadIdx.x & 31;
  uint32_t* ik = reinterpret_cast<uint32_t*>(m.keys);
  uint32_t* io = reinterpret_cast<uint32_t*>(m.out);
  for (int b = lane; b < 256; b += 32) m.bins[b] = 0u;
  __syncwarp();
  for (int j = lane; j < S; j += 32) {
    const uint32_t k = inner_key(half[j], j);
    ik[j] = k;
    atomicAdd(&m.bins[k >> InnerKeyOf<uint16_t>::top_shift], 1u);
  }
  __syncwarp();
  warp_topk_from<uint32_t>(ik, S, kin, io, m.bins, 0u, InnerKeyOf<uint16_t>::top_shift, true, 16);
  sort_desc_upto<uint32_t, 4>(io, kin);
  for (int r = lane; r < kin; r += 32) lst[r] = pack_inner(io[r]);
  __syncwarp();
}

// Key of the outer grid pair (p, q) of the packed lists: ord(fp32 sum) << 32 | ~flat.
__device__ __forceinline__ uint64_t packed_pair_key(const uint32_t* la, const uint32_t* lb, int p,
                                                    int q, int S) {
  const uint32_t ea = la[p], eb = lb[q];
  const float s = __fadd_rn(entry_value(ea), entry_value(eb));
  const uint32_t flat = entry_index(ea) * uint32_t(S) + entry_index(eb);
  return (uint64_t(ord_key(s)) << 32) | uint64_t(0xFFFFFFFFu - flat);
}

// Rare path of the outer selection: the top-K over every grid pair whose key reaches kth.
__device__ __noinline__ void packed_full_grid(const uint32_t* la, const uint32_t* lb, int S, int kin,
                                              int K, uint64_t kth, uint64_t* out, int kpad,
                                              uint32_t* hist) {
  auto grid_key = [&](int i, bool& valid) -> uint64_t {
    const uint64_t k = packed_pair_key(la, lb, i / kin, i % kin, S);
    valid = k >= kth;
    return k;
  };
  const uint64_t tau = radix_threshold(grid_key, kin * kin, K, 64, hist);
  collect_at_least(grid_key, kin * kin, tau, out, kpad);
}

// Exponent field of a packed entry's value, 1 for subnormals, 0 for zeros.
__device__ __forceinline__ uint32_t entry_exp(uint32_t e) {
  const uint32_t ex = (e >> 23) & 0xFFu;
  return (e & 0x7FFF0000u) == 0u ? 0u : (ex == 0u ? 1u : ex);
}

// Outer top-K over the staircase by bins of the sums' patterns (every staircase sum positive,
// lo = the smallest row-end sum's pattern, hi = the largest sum's).  Writes the K largest
// keys, in order, to out.  Returns false when a precondition does not hold.
__device__ bool outer_count(const CountSmem& m, const uint32_t* st, int cnt, int K, int kin, int S,
                            uint32_t lo, uint32_t hi) {
  const int lane = threadIdx.x & 31;
  if (hi - lo < 256u) return false;
  const int sh = (32 - __clz(int(hi - lo))) - 8;  // (hi - lo) >> sh < 256
  uint2* cand = reinterpret_cast<uint2*>(m.keys);
  uint32_t* bins = m.bins;
  const uint32_t junk = 256u + uint32_t(lane);
  reinterpret_cast<uint4*>(bins)[2 * lane] = make_uint4(0u, 0u, 0u, 0u);
  reinterpret_cast<uint4*>(bins)[2 * lane + 1] = make_uint4(0u, 0u, 0u, 0u);
  __syncwarp();
  for (int i = lane; i < cnt; i += 32) {
    const uint32_t pq = st[i];
    const uint32_t ea = m.la[pq >> 16], eb = m.lb[pq & 0xFFFFu];
    const uint32_t u = __float_as_uint(__fadd_rn(entry_value(ea), entry_value(eb)));
    cand[i] = make_uint2(u, entry_index(ea) * uint32_t(S) + entry_index(eb));
    bin_count(bins, 255u - ((u - lo) >> sh), junk);
  }
  __syncwarp();
  uint32_t above, bcnt;
  int bstar, ngroups;
  if (!count_scan(bins, K, m.groups, ngroups, bstar, above, bcnt)) return false;
  uint64_t* out = reinterpret_cast<uint64_t*>(m.out);
  uint64_t* tmp = reinterpret_cast<uint64_t*>(m.tmp);
  uint64_t* jslot = tmp + kBoundMax + lane;
  for (int i = lane; i < cnt; i += 32) {
    const uint2 x = cand[i];
    // key = (sum pattern | sign bit) << 32 | ~flat
    bin_place<uint64_t>(bins, 255u - ((x.x - lo) >> sh), uint32_t(bstar), junk, out, tmp, jslot,
                        (uint64_t(x.x | 0x80000000u) << 32) | uint64_t(~x.y));
  }
  __syncwarp();
  count_finish<uint64_t>(out, tmp, m.groups, ngroups, K, above, bcnt,
                         [](uint64_t x, uint64_t y) { return x > y; });
  return true;
}

// The general outer selection: radix select and sort on the staircase candidates' keys.
__device__ __noinline__ void outer_general(const CountSmem& m, const uint32_t* st, int cnt, int K,
                                           int S) {
  const int lane = threadIdx.x & 31;
  uint64_t* ck = reinterpret_cast<uint64_t*>(m.keys);
  uint64_t* out = reinterpret_cast<uint64_t*>(m.out);
  for (int i = lane; i < cnt; i += 32) {
    const uint32_t pq = st[i];
    ck[i] = packed_pair_key(m.la, m.lb, int(pq >> 16), int(pq & 0xFFFFu), S);
  }
  __syncwarp();
  warp_topk_from<uint64_t>(ck, cnt, K, out, m.bins, 0ull, -1, false);
  sort_desc_upto<uint64_t, 4>(out, K);
}

// The outer top-K of one task over the packed lists m.la, m.lb (each the top-kin of a half,
// in order): slots and scores, best first, to oi[0..K) and os[0..K).
__device__ void outer_task(const CountSmem& m, const uint32_t* st, int cnt, int K, int kin, int S,
                           int kpad, int32_t* oi, float* os) {
  const int lane = threadIdx.x & 31;
  uint64_t* out = reinterpret_cast<uint64_t*>(m.out);
  // The smallest row-end sum and the largest sum (both lists are in descending order),
  // and the exponent span of the lists' nonzero values.
  uint32_t lo = ~0u, emax = 0u, emin = 0xFFu;
  bool neg = false;
  for (int p = lane; p < kin; p += 32) {
    const float s = __fadd_rn(entry_value(m.la[p]), entry_value(m.lb[min(kin, K / (p + 1)) - 1]));
    neg = neg || !(s > 0.0f);
    lo = min(lo, __float_as_uint(s));
    const uint32_t xa = entry_exp(m.la[p]), xb = entry_exp(m.lb[p]);
    emax = max(emax, max(xa, xb));
    if (xa) emin = min(emin, xa);
    if (xb) emin = min(emin, xb);
  }
  lo = __reduce_min_sync(kFull, lo);
  emax = __reduce_max_sync(kFull, emax);
  emin = __reduce_min_sync(kFull, emin);
  const bool any_neg = __any_sync(kFull, neg);
  const uint32_t hi = __float_as_uint(__fadd_rn(entry_value(m.la[0]), entry_value(m.lb[0])));
  bool done = false;
  if (cnt > K && !any_neg) done = outer_count(m, st, cnt, K, kin, S, lo, hi);
  if (!done) outer_general(m, st, cnt, K, S);
  // Pairs right of the staircase that could still beat the K-th key: possible only when
  // fp32 rounding merges sums, i.e. when the values' exponents span more than 15.
  if (emax > emin + 15u) {
    const uint64_t kth = out[K - 1];
    const uint32_t kth_sum = uint32_t(kth >> 32);
    bool beyond = false;
    for (int p = lane; p < kin; p += 32) {
      for (int q = min(kin, K / (p + 1)); q < kin; ++q) {
        const uint64_t k = packed_pair_key(m.la, m.lb, p, q, S);
        if (uint32_t(k >> 32) < kth_sum) break;  // sums only fall along a row
        if (k > kth) beyond = true;
      }
    }
    if (__any_sync(kFull, beyond)) {
      packed_full_grid(m.la, m.lb, S, kin, K, kth, out, kpad, m.bins);
      sort_desc_upto<uint64_t, 4>(out, K);
    }
  }
  for (int r = lane; r < K; r += 32) {
    const uint64_t k = out[r];
    oi[r] = int32_t(0xFFFFFFFFu - uint32_t(k & 0xFFFFFFFFu));
    os[r] = ord_decode(uint32_t(k >> 32));
  }
  __syncwarp();
}

struct CountArgs {
  const void* kp;
  const void* qp;
  long long items;
  int Tc, T_total, t0;
  int S, W, R;
  int kin_max, kpad, cnt_w, cnt_r;
  int warps, tpw;
  size_t keys_bytes, per_warp;
  const uint32_t* stair_g;
  int32_t* idx_w;
  float* sc_w;
  int32_t* idx_r;
  float* sc_r;
};

// Selection tasks [task0, task1) of one warp (task = 2 * item + which; which 0: k' / top-W,
// 1: q' / top-R).
__device__ void count_tasks(const CountArgs& a, const uint32_t* stair_w, const uint32_t* stair_r,
                            unsigned char* wbase, long long task0, long long task1) {
  const int warp = threadIdx.x >> 5;
  const int S = a.S;
  const CountSmem m = count_smem(wbase + a.per_warp * warp, a.keys_bytes, a.kpad, a.kin_max);
  for (long long task = task0; task < task1; ++task) {
    const int which = int(task & 1);
    const long long wi = task >> 1;
    const long long item =
        a.Tc == a.T_total ? wi : (wi / a.Tc) * a.T_total + a.t0 + wi % a.Tc;
    const int K = which ? a.R : a.W;
    const int kin = min(K, S);
    const uint16_t* halves = static_cast<const uint16_t*>(which ? a.qp : a.kp) + item * 2 * S;

    // ---- 1. the top-kin of each half, packed, by (value desc, index asc) ----------------
    if (!inner_count(halves, S, kin, m, m.la)) inner_general(halves, S, kin, true, m, m.la);
    if (!inner_count(halves + S, S, kin, m, m.lb)) inner_general(halves + S, S, kin, true, m, m.lb);

    // ---- 2. top-K of the kin x kin grid of pair sums over the staircase -----------------
    outer_task(m, which ? stair_r : stair_w, which ? a.cnt_r : a.cnt_w, K, kin, S, a.kpad,
               (which ? a.idx_r : a.idx_w) + item * K, (which ? a.sc_r : a.sc_w) + item * K);
  }
}

__global__ void __launch_bounds__(128, 6) select_count_kernel(CountArgs a) {
  extern __shared__ __align__(16) unsigned char smem[];
  const uint32_t* stair_w;
  unsigned char* wbase;
  if (a.stair_g) {
    stair_w = a.stair_g;
    wbase = smem;
  } else {
    uint32_t* st = reinterpret_cast<uint32_t*>(smem);
    wbase = smem + (size_t(a.cnt_w + a.cnt_r) * 4 + 15) / 16 * 16;
    // warp 0's bins are free until its first task: scratch for the staircase scans
    int* tmp = reinterpret_cast<int*>(wbase + a.keys_bytes + size_t(a.kpad) * 8);
    build_stair(st, a.W, min(a.W, a.S), tmp);
    build_stair(st + a.cnt_w, a.R, min(a.R, a.S), tmp);
    stair_w = st;
  }
  const long long tasks = a.items * 2;
  const int warp = threadIdx.x >> 5;
  const long long task0 = ((long long)blockIdx.x * a.warps + warp) * a.tpw;
  const long long task1 = task0 + a.tpw < tasks ? task0 + a.tpw : tasks;
  count_tasks(a, stair_w, stair_w + a.cnt_w, wbase, task0, task1);
}

// The counting selection over a token window of bf16 halves, or SDM_EUNSUPPORTED when its
// limits do not hold (S % 8, S > kCountMaxS, W or R > kCountMaxK, fewer tasks than
// resident warps unless allow_small, shared memory).
int launch_select_count(const void* kp, const void* qp, const TokenWindow& win, int S, int W,
                        int R, int32_t* idx_w, float* sc_w, int32_t* idx_r, float* sc_r,
                        cudaStream_t s, const uint32_t* stair_g, bool allow_small) {
  const long long items = (long long)win.BH * win.Tc;
  if (items == 0) return SDM_OK;
  if (S % 8 || S > kCountMaxS || W > kCountMaxK || R > kCountMaxK) return SDM_EUNSUPPORTED;
  CountArgs a;
  a.kp = kp;
  a.qp = qp;
  a.items = items;
  a.Tc = win.Tc;
  a.T_total = win.T_total;
  a.t0 = win.t0;
  a.S = S;
  a.W = W;
  a.R = R;
  a.kin_max = max(min(W, S), min(R, S));
  const int kmax = max(W, R);
  a.kpad = 32;
  while (a.kpad < kmax) a.kpad <<= 1;
  a.cnt_w = stair_count(W, min(W, S));
  a.cnt_r = stair_count(R, min(R, S));
  a.idx_w = idx_w;
  a.sc_w = sc_w;
  a.idx_r = idx_r;
  a.sc_r = sc_r;
  a.keys_bytes = select_key_bytes(a.kpad, S, max(a.cnt_w, a.cnt_r), 4);
  a.per_warp = (count_per_warp_bytes(a.keys_bytes, a.kpad, a.kin_max) + 15) / 16 * 16;
  a.stair_g = stair_g;
  const size_t stair_bytes = stair_g ? 0 : (size_t(a.cnt_w + a.cnt_r) * 4 + 15) / 16 * 16;
  int dev = 0, max_smem = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return SDM_ECUDA;
  const int warps = 4;
  const size_t smem = stair_bytes + a.per_warp * warps;
  if (smem > size_t(max_smem)) return SDM_EUNSUPPORTED;
  a.warps = warps;
  const void* fn = reinterpret_cast<const void*>(&select_count_kernel);
  // The whole shared-memory carveout: six blocks fit beside each other only with it.
  if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)) != cudaSuccess ||
      cudaFuncSetAttribute(fn, cudaFuncAttributePreferredSharedMemoryCarveout,
                           int(cudaSharedmemCarveoutMaxShared)) != cudaSuccess)
    return SDM_ECUDA;
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, warps * 32, smem) != cudaSuccess)
    return SDM_ECUDA;
  const long long tasks = items * 2;
  const long long resident = (long long)sms * (per_sm > 0 ? per_sm : 1) * warps;
  // With fewer tasks than warp slots the general path's warp pairs finish sooner.
  if (!allow_small && tasks < resident) return SDM_EUNSUPPORTED;
  long long tpw = tasks / (resident * 64);
  tpw = tpw < 1 ? 1 : (tpw > 64 ? 64 : tpw);
  a.tpw = int(tpw);
  const long long blocks = (tasks + warps * tpw - 1) / (warps * tpw);
  if (blocks > 0x7FFFFFFFLL) return SDM_EUNSUPPORTED;
  void* args[] = {&a};
  if (cudaLaunchKernel(fn, dim3(unsigned(blocks)), dim3(warps * 32), args, smem, s) != cudaSuccess)
    return SDM_ECUDA;
  return last_launch_status();
}

}  // namespace
}  // namespace sdm
