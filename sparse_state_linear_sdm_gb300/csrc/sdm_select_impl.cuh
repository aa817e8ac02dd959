// Product-key slot selection (Sparse Delta Memory technical summary,
// gist.science/it/paper/2607.07386, "Meccanismo Core" item 2):
// topk(s1 (+) s2) = topk(topk(s1) (+) topk(s2)) without forming the N slot scores.
//
// One warp owns one (b, h, t, k'-or-q') task:
//   1. each half (S sub-scores) -> its top-k, k = min(K, S), ranked by
//      (value desc, index asc): warp radix select on a composite integer key
//      (order-preserving value bits, then S-1-index), then a warp bitonic sort;
//   2. outer top-K over the k x k grid of fp32 sums, ranked by (sum desc, flat asc)
//      with flat = i*S + j.  Only the "staircase" (p+1)(q+1) <= K of the two sorted
//      lists is scanned: every other pair is dominated by at least K pairs in exact
//      arithmetic.  Because fp32 rounding can merge sums (and the flat tie-break
//      need not follow the list ranks), the kernel then walks each row past the
//      staircase while the sum can still reach the K-th key; if any pair there beats
//      it, the selection is redone over every grid pair that can, so the result is
//      always exactly the top-K of the full grid.
// No tensor cores: this is compare/select work on CUDA cores.
#pragma once

#include "sdm_internal.cuh"

namespace sdm {
namespace {

constexpr unsigned kFull = 0xFFFFFFFFu;

// Order-preserving map of an fp32 value to uint32 (larger value -> larger key);
// -0 maps like +0 so the two tie on value.
__device__ __forceinline__ uint32_t ord_key(float x) {
  uint32_t u = __float_as_uint(x);
  if ((u & 0x7FFFFFFFu) == 0u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float ord_decode(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// Warp-cooperative radix select.  key_of(i, valid) yields a distinct key for each
// valid i in [0, n).  Returns tau such that exactly `need` valid keys are >= tau.
// `bits` (multiple of 8) is the key width; hist is 256 warp-private counters.
template <class KeyOf>
__device__ uint64_t radix_threshold(const KeyOf& key_of, int n, int need, int bits,
                                    uint32_t* hist) {
  const int lane = threadIdx.x & 31;
  uint64_t prefix = 0;
  for (int shift = bits - 8; shift >= 0; shift -= 8) {
    const uint64_t hi_mask = (shift + 8 >= 64) ? 0ull : (~0ull << (shift + 8));
    for (int b = lane; b < 256; b += 32) hist[b] = 0u;
    __syncwarp();
    for (int i = lane; i < n; i += 32) {
      bool valid;
      const uint64_t k = key_of(i, valid);
      if (valid && (k & hi_mask) == prefix) atomicAdd(&hist[(k >> shift) & 255u], 1u);
    }
    __syncwarp();
    // Bins scanned from the top: lane l owns bins 255-8l ... 248-8l.
    uint32_t c[8];
    uint32_t s = 0;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      c[k] = hist[255 - 8 * lane - k];
      s += c[k];
    }
    uint32_t incl = s;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const uint32_t y = __shfl_up_sync(kFull, incl, off);
      if (lane >= off) incl += y;
    }
    const uint32_t excl = incl - s;
    const bool mine = excl < uint32_t(need) && uint32_t(need) <= incl;
    const int src = __ffs(__ballot_sync(kFull, mine)) - 1;
    int digit = 0;
    uint32_t above = 0, cnt = 0;
    if (mine) {
      uint32_t run = excl;
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        if (cnt == 0u && run + c[k] >= uint32_t(need)) {
          digit = 255 - 8 * lane - k;
          above = run;
          cnt = c[k];
        }
        run += c[k];
      }
    }
    digit = __shfl_sync(kFull, digit, src);
    above = __shfl_sync(kFull, above, src);
    cnt = __shfl_sync(kFull, cnt, src);
    prefix |= uint64_t(digit) << shift;
    need -= int(above);
    __syncwarp();
    if (cnt == uint32_t(need)) break;  // the whole bucket is in: done
  }
  return prefix;
}

// Writes the valid keys >= tau to out[0..cap), in index order (never past cap).
// Returns how many keys were >= tau.
template <class KeyOf>
__device__ int collect_at_least(const KeyOf& key_of, int n, uint64_t tau, uint64_t* out, int cap) {
  const int lane = threadIdx.x & 31;
  int base = 0;
  for (int i0 = 0; i0 < n; i0 += 32) {
    const int i = i0 + lane;
    bool valid = false;
    uint64_t k = 0;
    if (i < n) k = key_of(i, valid);
    const bool sel = valid && k >= tau;
    const unsigned m = __ballot_sync(kFull, sel);
    const int pos = base + __popc(m & ((1u << lane) - 1u));
    if (sel && pos < cap) out[pos] = k;
    base += __popc(m);
  }
  __syncwarp();
  return base;
}

// Bucket search over a 256-bin digit histogram, from the top: the digit d with
// above < need <= above + cnt, where above counts digits > d and cnt = hist[d].
__device__ __forceinline__ void find_bucket(const uint32_t* hist, int need, int& digit,
                                            uint32_t& above, uint32_t& cnt) {
  const int lane = threadIdx.x & 31;
  uint32_t c[8];
  uint32_t s = 0;
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    c[k] = hist[255 - 8 * lane - k];  // lane l owns bins 255-8l ... 248-8l
    s += c[k];
  }
  uint32_t incl = s;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const uint32_t y = __shfl_up_sync(kFull, incl, off);
    if (lane >= off) incl += y;
  }
  const uint32_t excl = incl - s;
  const bool mine = excl < uint32_t(need) && uint32_t(need) <= incl;
  const int src = __ffs(__ballot_sync(kFull, mine)) - 1;
  int d = 0;
  uint32_t ab = 0, ct = 0;
  if (mine) {
    uint32_t run = excl;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      if (ct == 0u && run + c[k] >= uint32_t(need)) {
        d = 255 - 8 * lane - k;
        ab = run;
        ct = c[k];
      }
      run += c[k];
    }
  }
  digit = __shfl_sync(kFull, d, src);
  above = __shfl_sync(kFull, ab, src);
  cnt = __shfl_sync(kFull, ct, src);
}

template <typename Key>
__device__ __forceinline__ void warp_minmax(Key& mx, Key& mn) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const Key a = __shfl_xor_sync(kFull, mx, off), b = __shfl_xor_sync(kFull, mn, off);
    mx = a > mx ? a : mx;
    mn = b < mn ? b : mn;
  }
}

// Bits needed to hold `range` (0 for 0).
template <typename Key>
__device__ __forceinline__ int bit_length(Key range) {
  return int(sizeof(Key) * 8) -
         (sizeof(Key) == 8 ? __clzll((long long)range) : __clz(int(uint32_t(range))));
}

// Selects the `need` largest of the n distinct keys in buf[0..n) and writes them,
// unordered, to out[0..need).  MSB-first radix select on the offset (key - base) with
// 8-bit digits d = (key - base) >> shift: each pass keeps only the bucket that holds the
// need-th largest (compacted in place in buf) and narrows the window by 8 bits, so only
// the first pass touches all n keys; a bucket of at most 32 keys is finished by ranking
// its keys against each other.  shift < 0: base and shift are fitted to the keys'
// range first.  With hist_ready the first pass's histogram is already in hist.
// tie_shift >= 0 declares that the key bits below tie_shift are a position written so
// that, among keys equal above it, larger keys come earlier in buf (and base is a
// multiple of 1 << tie_shift): once a pass at that shift leaves a bucket of keys equal
// above it, its first `need` keys are the largest and the search stops there.
template <typename Key>
__device__ void warp_topk_from(Key* buf, int n, int need, Key* out, uint32_t* hist, Key base,
                               int shift, bool hist_ready, int tie_shift = -1) {
  const int lane = threadIdx.x & 31;
  if (need >= n) {
    for (int i = lane; i < n; i += 32) out[i] = buf[i];
    __syncwarp();
    return;
  }
  if (shift < 0) {
    Key mx = 0, mn = ~Key(0);
    for (int i = lane; i < n; i += 32) {
      const Key k = buf[i];
      mx = k > mx ? k : mx;
      mn = k < mn ? k : mn;
    }
    warp_minmax(mx, mn);
    base = mn;
    const int bits = bit_length<Key>(mx - mn);
    shift = bits > 8 ? bits - 8 : 0;
    hist_ready = false;
  }
  int n_out = 0;
  for (;;) {
    if (!hist_ready) {
      for (int b = lane; b < 256; b += 32) hist[b] = 0u;
      __syncwarp();
      for (int i = lane; i < n; i += 32) atomicAdd(&hist[unsigned((buf[i] - base) >> shift)], 1u);
      __syncwarp();
    }
    hist_ready = false;
    int digit;
    uint32_t above, cnt;
    find_bucket(hist, need, digit, above, cnt);
    // Keys above the bucket are final; the bucket is compacted to the front of buf.
    int base_up = n_out, base_eq = 0;
    for (int i0 = 0; i0 < n; i0 += 32) {
      const int i = i0 + lane;
      Key k = 0;
      int dg = -1;
      if (i < n) {
        k = buf[i];
        dg = int((k - base) >> shift);
      }
      const bool up = dg > digit, eq = dg == digit;
      const unsigned mu = __ballot_sync(kFull, up), me = __ballot_sync(kFull, eq);
      const unsigned lt = (1u << lane) - 1u;
      if (up) out[base_up + __popc(mu & lt)] = k;
      if (eq) buf[base_eq + __popc(me & lt)] = k;  // positions <= i: already read
      base_up += __popc(mu);
      base_eq += __popc(me);
      __syncwarp();
    }
    n_out += int(above);
    need -= int(above);
    n = int(cnt);
    if (n == need || shift == tie_shift) {
      // The bucket keeps buf's order (the compaction is stable).
      for (int i = lane; i < need; i += 32) out[n_out + i] = buf[i];
      __syncwarp();
      return;
    }
    if (n <= 32) {
      // Small bucket: rank its (distinct) keys directly, one per lane, instead of more
      // 8-bit passes (ties in value or sum leave only index bits to resolve).
      const Key mine = lane < n ? buf[lane] : Key(0);
      int rank = 0;
      for (int j = 0; j < n; ++j) {
        const Key kj = __shfl_sync(kFull, mine, j);
        rank += kj > mine ? 1 : 0;
      }
      if (lane < n && rank < need) out[n_out + rank] = mine;
      __syncwarp();
      return;
    }
    // >= 2 distinct keys share the digit, so the window is wider than one key: narrow it.
    base += Key(digit) << shift;
    shift = shift >= 8 ? shift - 8 : 0;
  }
}

// Compare-exchange of registers e and e ^ JE (JE = partner distance / 32) in one
// bitonic step of block size k.
template <typename Key, int E, int JE>
__device__ __forceinline__ void cx_regs(Key (&v)[E], int k, int lane) {
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const int ep = e ^ JE;
    if (ep > e) {
      const bool desc = ((e * 32 + lane) & k) == 0;
      const Key a = v[e], b = v[ep];
      if (desc ? (a < b) : (a > b)) {
        v[e] = b;
        v[ep] = a;
      }
    }
  }
}

// Bitonic sort (descending) of buf[0..count) padded with zero keys to 32*E entries.
// Element i lives in lane i % 32, register i / 32.  The stage loops stay rolled (small
// code); only the per-register work of a step is unrolled.
template <typename Key, int E>
__device__ __noinline__ void sort_desc(Key* buf, int count) {
  const int lane = threadIdx.x & 31;
  Key v[E];
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const int i = e * 32 + lane;
    v[e] = i < count ? buf[i] : Key(0);
  }
  constexpr int n = 32 * E;
#pragma unroll 1
  for (int k = 2; k <= n; k <<= 1) {
#pragma unroll 1
    for (int j = k >> 1; j > 0; j >>= 1) {
      if (j >= 32) {
        if (E >= 2 && j == 32) cx_regs<Key, E, (E >= 2 ? 1 : 0)>(v, k, lane);
        else if (E >= 4 && j == 64) cx_regs<Key, E, (E >= 4 ? 2 : 0)>(v, k, lane);
        else if (E >= 8 && j == 128) cx_regs<Key, E, (E >= 8 ? 4 : 0)>(v, k, lane);
        else if (E >= 16 && j == 256) cx_regs<Key, E, (E >= 16 ? 8 : 0)>(v, k, lane);
        else if (E >= 32 && j == 512) cx_regs<Key, E, (E >= 32 ? 16 : 0)>(v, k, lane);
      } else {
        const bool lower = (lane & j) == 0;
#pragma unroll
        for (int e = 0; e < E; ++e) {
          const Key other = __shfl_xor_sync(kFull, v[e], j);
          const bool desc = ((e * 32 + lane) & k) == 0;
          const bool keep_max = (lower == desc);
          v[e] = keep_max ? (v[e] > other ? v[e] : other) : (v[e] < other ? v[e] : other);
        }
      }
    }
  }
  __syncwarp();
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const int i = e * 32 + lane;
    if (i < count) buf[i] = v[e];
  }
  __syncwarp();
}

template <typename Key, int EMAX>
__device__ void sort_desc_upto(Key* buf, int count) {
  if (count <= 32) sort_desc<Key, 1>(buf, count);
  else if (count <= 64 || EMAX < 4) sort_desc<Key, (EMAX < 2 ? EMAX : 2)>(buf, count);
  else if (count <= 128 || EMAX < 8) sort_desc<Key, (EMAX < 4 ? EMAX : 4)>(buf, count);
  else if (count <= 256 || EMAX < 16) sort_desc<Key, (EMAX < 8 ? EMAX : 8)>(buf, count);
  else if (count <= 512 || EMAX < 32) sort_desc<Key, (EMAX < 16 ? EMAX : 16)>(buf, count);
  else sort_desc<Key, EMAX>(buf, count);
}

__host__ __device__ inline int imin(int a, int b) { return a < b ? a : b; }

__host__ __device__ inline int stair_count(int K, int kin) {
  int c = 0;
  for (int p = 0; p < kin; ++p) c += imin(kin, K / (p + 1));
  return c;
}

// bf16 halves use 32-bit keys (16 value bits, 16 index bits); fp32 halves 48-bit keys
// (32 value bits, 16 index bits) held in 64 bits.
template <typename Tin>
struct InnerKeyOf {
  using type = uint64_t;
  static constexpr int top_shift = 40;  // shift of the key's top value byte
};
template <>
struct InnerKeyOf<uint16_t> {
  using type = uint32_t;
  static constexpr int top_shift = 24;
};

__device__ __forceinline__ uint32_t inner_key(uint16_t u, int j) {
  uint32_t b = u;
  if ((b & 0x7FFFu) == 0u) b = 0u;  // -0 ranks as +0
  const uint32_t o = (b & 0x8000u) ? (~b & 0xFFFFu) : (b | 0x8000u);
  return (o << 16) | (0xFFFFu - uint32_t(j));
}
__device__ __forceinline__ uint64_t inner_key(float x, int j) {
  return (uint64_t(ord_key(x)) << 16) | uint64_t(0xFFFFu - uint32_t(j));
}
__device__ __forceinline__ float inner_value(uint32_t key) {
  const uint32_t o = key >> 16;
  const uint32_t b = (o & 0x8000u) ? (o & 0x7FFFu) : (~o & 0xFFFFu);
  return __uint_as_float(b << 16);
}
__device__ __forceinline__ float inner_value(uint64_t key) {
  return ord_decode(uint32_t(key >> 16));
}

// Unpacks one 16-byte vector of sub-scores.
template <typename Tin>
__device__ __forceinline__ void unpack16(const uint4& q, float* v);
template <>
__device__ __forceinline__ void unpack16<uint16_t>(const uint4& q, float* v) {
  const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[2 * i] = __uint_as_float(w[i] << 16);
    v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}
template <>
__device__ __forceinline__ void unpack16<float>(const uint4& q, float* v) {
  v[0] = __uint_as_float(q.x);
  v[1] = __uint_as_float(q.y);
  v[2] = __uint_as_float(q.z);
  v[3] = __uint_as_float(q.w);
}
__device__ __forceinline__ uint32_t inner_key_f(float v, int j, uint32_t*) {
  return inner_key(uint16_t(__float_as_uint(v) >> 16), j);
}
__device__ __forceinline__ uint64_t inner_key_f(float v, int j, uint64_t*) { return inner_key(v, j); }

// Keys of one half into ik[0..S) with the histogram of their top value byte: 16-byte
// loads when every half is 16-byte aligned (vec), element loads otherwise.
template <typename Tin>
__device__ __forceinline__ void load_half_keys(const Tin* src, int S, bool vec,
                                               typename InnerKeyOf<Tin>::type* ik, uint32_t* hist) {
  using IKey = typename InnerKeyOf<Tin>::type;
  constexpr int EPV = 16 / int(sizeof(Tin));
  constexpr int TOP = InnerKeyOf<Tin>::top_shift;
  const int lane = threadIdx.x & 31;
  for (int b = lane; b < 256; b += 32) hist[b] = 0u;
  __syncwarp();
  if (vec) {
    // Up to four 16-byte loads per lane are issued before any is used, so their
    // latencies overlap instead of adding up.
    constexpr int UNR = 4;
    const uint4* src4 = reinterpret_cast<const uint4*>(src);
    const int nvec = S / EPV;
    for (int c0 = lane; c0 < nvec; c0 += 32 * UNR) {
      uint4 q[UNR];
#pragma unroll
      for (int u = 0; u < UNR; ++u)
        q[u] = c0 + 32 * u < nvec ? __ldg(src4 + c0 + 32 * u) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
      for (int u = 0; u < UNR; ++u) {
        const int c = c0 + 32 * u;
        if (c >= nvec) break;
        float f[EPV];
        unpack16<Tin>(q[u], f);
        IKey k[EPV];
#pragma unroll
        for (int i = 0; i < EPV; ++i) {
          k[i] = inner_key_f(f[i], c * EPV + i, static_cast<IKey*>(nullptr));
          atomicAdd(&hist[unsigned(k[i] >> TOP) & 255u], 1u);
        }
        uint4* dst = reinterpret_cast<uint4*>(ik + c * EPV);
#pragma unroll
        for (int w = 0; w < int(EPV * sizeof(IKey) / 16); ++w) dst[w] = reinterpret_cast<const uint4*>(k)[w];
      }
    }
  } else {
    for (int j = lane; j < S; j += 32) {
      const IKey k = inner_key(src[j], j);
      ik[j] = k;
      atomicAdd(&hist[unsigned(k >> TOP) & 255u], 1u);
    }
  }
  __syncwarp();
}

// Shared memory of one warp: key buffer (one half, its bucket, or the staircase
// candidates), the selected keys, the histogram and the two inner lists.
__host__ __device__ inline size_t select_key_bytes(int kpad, int S, int cnt_max, int inner_key_bytes) {
  size_t keys = size_t(S) * inner_key_bytes;
  if (size_t(cnt_max) * 8 > keys) keys = size_t(cnt_max) * 8;
  return (keys + 15) / 16 * 16;
}

__host__ __device__ inline size_t select_per_warp_bytes(int kpad, int kin_max, int S, int cnt_max,
                                                        int inner_key_bytes) {
  size_t keys = select_key_bytes(kpad, S, cnt_max, inner_key_bytes);
  keys = (keys + 15) / 16 * 16;
  const size_t b = keys + size_t(kpad) * 8 + 256 * 4 + size_t(kin_max) * 16;
  return (b + 15) / 16 * 16;
}

struct SelectArgs {
  const void* kp;
  const void* qp;
  long long items;     // (b, h, t) triples of the token window: BH * Tc
  int Tc, T_total, t0;  // window tokens [t0, t0 + Tc) of sequences of T_total tokens
  int S, W, R;
  int kin_max;   // max(min(W,S), min(R,S))
  int kpad;      // max(W, R, 32) rounded up to a power of two (selected-key buffer)
  int cnt_w, cnt_r;
  int warps;
  int tpw;            // consecutive tasks per warp (per warp pair in pair mode)
  size_t keys_bytes;  // per-warp key buffer
  bool vec;           // every half starts on a 16-byte boundary
  const uint32_t* stair_g;  // both staircases prebuilt in device memory (write, then read),
                            // or nullptr: every block builds them in its shared memory
  int32_t* idx_w;
  float* sc_w;
  int32_t* idx_r;
  float* sc_r;
};

// Fills the staircase {(p, q): p, q < kin, (p+1)(q+1) <= K} as p << 16 | q, row by row.
// Each thread owns a run of rows; their offsets come from a block-wide prefix sum of the
// row lengths.  tmp: one word per warp of the block.  Ends with a block barrier.
__device__ void build_stair(uint32_t* st, int K, int kin, int* tmp) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int per = (kin + int(blockDim.x) - 1) / int(blockDim.x);
  const int p0 = min(kin, tid * per), p1 = min(kin, p0 + per);
  int mine = 0;
  for (int p = p0; p < p1; ++p) mine += min(kin, K / (p + 1));
  int incl = mine;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int y = __shfl_up_sync(kFull, incl, off);
    if (lane >= off) incl += y;
  }
  if (lane == 31) tmp[warp] = incl;
  __syncthreads();
  int off = incl - mine;
  for (int w = 0; w < warp; ++w) off += tmp[w];
  for (int p = p0; p < p1; ++p) {
    const int len = min(kin, K / (p + 1));
    for (int q = 0; q < len; ++q) st[off + q] = (uint32_t(p) << 16) | uint32_t(q);
    off += len;
  }
  __syncthreads();
}

// Rare path of the outer selection (needs rounding merges or massive ties): the top-K
// over every grid pair whose key reaches `kth` (the staircase's K-th key), into out.
__device__ __noinline__ void outer_full_grid(const float* aval, const float* bval,
                                             const int32_t* aidx, const int32_t* bidx, int S,
                                             int kin, int K, uint64_t kth, uint64_t* out, int kpad,
                                             uint32_t* hist) {
  auto grid_key = [&](int i, bool& valid) -> uint64_t {
    const int p = i / kin, q = i % kin;
    const float s = __fadd_rn(aval[p], bval[q]);
    const uint32_t flat = uint32_t(aidx[p]) * uint32_t(S) + uint32_t(bidx[q]);
    const uint64_t k = (uint64_t(ord_key(s)) << 32) | uint64_t(0xFFFFFFFFu - flat);
    valid = k >= kth;
    return k;
  };
  const uint64_t tau2 = radix_threshold(grid_key, kin * kin, K, 64, hist);
  collect_at_least(grid_key, kin * kin, tau2, out, kpad);
}

// Shared memory of a selecting block: the two staircases, then one region per warp.
struct SelectSmem {
  uint32_t* stair_w;
  uint32_t* stair_r;
  unsigned char* wbase;
  size_t per_warp;  // bytes of one warp's region (16-byte multiple)
};

__device__ __forceinline__ SelectSmem select_smem(const SelectArgs& a, unsigned char* smem) {
  SelectSmem m;
  if (a.stair_g) {
    m.stair_w = const_cast<uint32_t*>(a.stair_g);
    m.stair_r = m.stair_w + a.cnt_w;
    m.wbase = smem;
  } else {
    m.stair_w = reinterpret_cast<uint32_t*>(smem);
    m.stair_r = m.stair_w + a.cnt_w;
    m.wbase = smem + (size_t(a.cnt_w + a.cnt_r) * 4 + 15) / 16 * 16;
  }
  const size_t per_warp = a.keys_bytes + size_t(a.kpad) * 8 + 256 * 4 + size_t(a.kin_max) * 16;
  m.per_warp = (per_warp + 15) / 16 * 16;
  return m;
}

// Both staircases, built by every thread of the block (ends with a block barrier).  Warp 0's
// histogram is free until its first task: scratch for the staircase scans.
__device__ __forceinline__ void select_build_stairs(const SelectArgs& a, const SelectSmem& m) {
  int* tmp = reinterpret_cast<int*>(m.wbase + a.keys_bytes + size_t(a.kpad) * 8);
  build_stair(m.stair_w, a.W, min(a.W, a.S), tmp);
  build_stair(m.stair_r, a.R, min(a.R, a.S), tmp);
}

// Selection tasks [task0, task1) (task = 2 * item + which, which 0: k' / top-W, 1: q' /
// top-R) by one warp (PAIR false) or by the warp pair `unit` (PAIR true: warps 2*unit and
// 2*unit + 1 of the block, one half each, joined by named barrier 1 + unit).
template <typename Tin, int EMAX, bool PAIR>
__device__ void select_tasks(const SelectArgs& a, const SelectSmem& m, long long task0,
                             long long task1) {
  using IKey = typename InnerKeyOf<Tin>::type;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int S = a.S;
  unsigned char* wp = m.wbase + m.per_warp * warp;
  unsigned char* keys = wp;
  uint64_t* out = reinterpret_cast<uint64_t*>(wp + a.keys_bytes);
  uint32_t* hist = reinterpret_cast<uint32_t*>(out + a.kpad);
  // Pair mode: warps 2u and 2u+1 share a task; the inner lists live in warp 2u's region.
  const int role = PAIR ? (warp & 1) : 0;
  const int unit = PAIR ? (warp >> 1) : warp;
  unsigned char* lp = PAIR ? m.wbase + m.per_warp * (warp & ~1) : wp;
  float* aval = reinterpret_cast<float*>(lp + a.keys_bytes + size_t(a.kpad) * 8 + 256 * 4);
  float* bval = aval + a.kin_max;
  int32_t* aidx = reinterpret_cast<int32_t*>(bval + a.kin_max);
  int32_t* bidx = aidx + a.kin_max;
  const uint32_t* stair_w = m.stair_w;
  const uint32_t* stair_r = m.stair_r;
  for (long long task = task0; task < task1; ++task) {
    const int which = int(task & 1);
    // (b, h, t) triple in the full [B, H, T_total] arrays
    const long long wi = task >> 1;
    const long long item =
        a.Tc == a.T_total ? wi : (wi / a.Tc) * a.T_total + a.t0 + wi % a.Tc;
    const int K = which ? a.R : a.W;
    const int kin = min(K, S);
    const Tin* halves = static_cast<const Tin*>(which ? a.qp : a.kp) + item * 2 * S;

    // ---- 1. top-kin of each half, ranked by (value desc, index asc) ---------------
    for (int h = role; h < (PAIR ? role + 1 : 2); ++h) {
      IKey* ik = reinterpret_cast<IKey*>(keys);
      IKey* io = reinterpret_cast<IKey*>(out);
      load_half_keys<Tin>(halves + (long long)h * S, S, a.vec, ik, hist);
      // ik is in index order and the low 16 key bits are 0xFFFF - index: equal values
      // are already ranked by position once the value bits are resolved.
      warp_topk_from<IKey>(ik, S, kin, io, hist, IKey(0), InnerKeyOf<Tin>::top_shift, true, 16);
      sort_desc_upto<IKey, EMAX>(io, kin);
      float* dv = h ? bval : aval;
      int32_t* di = h ? bidx : aidx;
      for (int r = lane; r < kin; r += 32) {
        const IKey k = io[r];
        dv[r] = inner_value(k);
        di[r] = min(int(0xFFFFu - uint32_t(k & 0xFFFFu)), S - 1);
      }
      __syncwarp();
    }

    if (PAIR) {  // both halves' lists are in place; the second warp waits for the next task
      asm volatile("bar.sync %0, 64;" ::"r"(1 + unit) : "memory");
      if (role) {
        asm volatile("bar.sync %0, 64;" ::"r"(1 + unit) : "memory");
        continue;
      }
    }

    // ---- 2. top-K of the kin x kin grid of pair sums -------------------------------
    const uint32_t* st = which ? stair_r : stair_w;
    const int cnt = which ? a.cnt_r : a.cnt_w;
    auto pair_key = [&](int p, int q) -> uint64_t {
      const float s = __fadd_rn(aval[p], bval[q]);
      const uint32_t flat = uint32_t(aidx[p]) * uint32_t(S) + uint32_t(bidx[q]);
      return (uint64_t(ord_key(s)) << 32) | uint64_t(0xFFFFFFFFu - flat);
    };
    uint64_t* ck = reinterpret_cast<uint64_t*>(keys);
    int shift = 0;
    uint64_t base = 0;
    if (cnt > K) {
      // Digit window: (0, 0) has the largest sum and some row end the smallest (sums fall
      // along rows and columns).  The flat tie-break can order keys of equal sums either
      // way, so the window spans those sums with every flat: no key falls outside it.
      uint32_t lo = ~0u;
      for (int p = lane; p < kin; p += 32) {
        const uint32_t k = ord_key(__fadd_rn(aval[p], bval[min(kin, K / (p + 1)) - 1]));
        lo = k < lo ? k : lo;
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        const uint32_t o = __shfl_xor_sync(kFull, lo, off);
        lo = o < lo ? o : lo;
      }
      const uint64_t mx = (uint64_t(ord_key(__fadd_rn(aval[0], bval[0]))) << 32) | 0xFFFFFFFFull;
      base = uint64_t(lo) << 32;
      const int bits = bit_length<uint64_t>(mx - base);
      shift = bits > 8 ? bits - 8 : 0;
      for (int b = lane; b < 256; b += 32) hist[b] = 0u;
      __syncwarp();
    }
    for (int c = lane; c < cnt; c += 32) {
      const uint32_t pq = st[c];
      const uint64_t k = pair_key(int(pq >> 16), int(pq & 0xFFFFu));
      ck[c] = k;
      if (cnt > K) atomicAdd(&hist[unsigned((k - base) >> shift)], 1u);
    }
    __syncwarp();
    warp_topk_from<uint64_t>(ck, cnt, K, out, hist, base, shift, true);
    sort_desc_upto<uint64_t, EMAX>(out, K);
    const uint64_t kth = out[K - 1];
    const uint32_t kth_sum = uint32_t(kth >> 32);
    // Pairs right of the staircase that could still beat the K-th key.
    bool beyond = false;
    for (int p = lane; p < kin; p += 32) {
      for (int q = min(kin, K / (p + 1)); q < kin; ++q) {
        const uint64_t k = pair_key(p, q);
        if (uint32_t(k >> 32) < kth_sum) break;  // sums only fall along a row
        if (k > kth) beyond = true;
      }
    }
    if (__any_sync(kFull, beyond)) {
      outer_full_grid(aval, bval, aidx, bidx, S, kin, K, kth, out, a.kpad, hist);
      sort_desc_upto<uint64_t, EMAX>(out, K);
    }
    int32_t* oi = (which ? a.idx_r : a.idx_w) + item * K;
    float* os = (which ? a.sc_r : a.sc_w) + item * K;
    for (int r = lane; r < K; r += 32) {
      const uint64_t k = out[r];
      oi[r] = int32_t(0xFFFFFFFFu - uint32_t(k & 0xFFFFFFFFu));
      os[r] = ord_decode(uint32_t(k >> 32));
    }
    __syncwarp();
    if (PAIR) asm volatile("bar.sync %0, 64;" ::"r"(1 + unit) : "memory");  // lists free again
  }
}

template <typename Tin, int EMAX, bool PAIR>
__global__ void __launch_bounds__(128) select_kernel(SelectArgs a) {
  extern __shared__ __align__(16) unsigned char smem[];
  const SelectSmem m = select_smem(a, smem);
  if (!a.stair_g) select_build_stairs(a, m);
  // A short run of consecutive tasks per warp (no persistent grid): blocks that start
  // late, e.g. behind a kernel on another stream, do not hold up the others.
  const long long tasks = a.items * 2;
  const int warp = threadIdx.x >> 5;
  const int unit = PAIR ? (warp >> 1) : warp;
  const int units = PAIR ? a.warps / 2 : a.warps;
  const long long task0 = ((long long)blockIdx.x * units + unit) * a.tpw;
  const long long task1 = task0 + a.tpw < tasks ? task0 + a.tpw : tasks;
  select_tasks<Tin, EMAX, PAIR>(a, m, task0, task1);
}

// Arguments and shared-memory sizes of a selection over a token window (warps, tpw and
// the launch shape are left to the caller).  stair_bytes: both staircases; per_warp: one
// warp's region.
template <typename Tin>
void select_args(const void* kp, const void* qp, const TokenWindow& win, int S, int W, int R,
                 int32_t* idx_w, float* sc_w, int32_t* idx_r, float* sc_r, SelectArgs* out,
                 size_t* stair_bytes, size_t* per_warp_bytes) {
  constexpr bool kBf16 = sizeof(Tin) == 2;
  SelectArgs a;
  a.kp = kp;
  a.qp = qp;
  a.items = (long long)win.BH * win.Tc;
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
  const int ikb = kBf16 ? 4 : 8;
  a.keys_bytes = select_key_bytes(a.kpad, S, max(a.cnt_w, a.cnt_r), ikb);
  a.vec = (S * int(sizeof(Tin))) % 16 == 0;
  a.warps = 0;
  a.tpw = 1;
  a.stair_g = nullptr;
  *stair_bytes = (size_t(a.cnt_w + a.cnt_r) * 4 + 15) / 16 * 16;
  *per_warp_bytes = select_per_warp_bytes(a.kpad, a.kin_max, S, max(a.cnt_w, a.cnt_r), ikb);
  *out = a;
}

template <typename Tin>
int launch_select_t(const void* kp, const void* qp, const TokenWindow& win, int S, int W, int R,
                    int32_t* idx_w, float* sc_w, int32_t* idx_r, float* sc_r, cudaStream_t s,
                    const uint32_t* stair_g) {
  constexpr bool kBf16 = sizeof(Tin) == 2;
  const long long items = (long long)win.BH * win.Tc;
  if (items == 0) return SDM_OK;
  SelectArgs a;
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
  const int ikb = kBf16 ? 4 : 8;
  a.keys_bytes = select_key_bytes(a.kpad, S, max(a.cnt_w, a.cnt_r), ikb);
  a.stair_g = stair_g;
  const size_t stair_bytes = stair_g ? 0 : (size_t(a.cnt_w + a.cnt_r) * 4 + 15) / 16 * 16;
  const size_t per_warp = select_per_warp_bytes(a.kpad, a.kin_max, S, max(a.cnt_w, a.cnt_r), ikb);
  int dev = 0, max_smem = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return SDM_ECUDA;
  int warps = 4;
  while (warps > 1 && stair_bytes + per_warp * warps > size_t(max_smem)) --warps;
  if (stair_bytes + per_warp * warps > size_t(max_smem)) return SDM_EUNSUPPORTED;
  a.warps = warps;
  const size_t smem = stair_bytes + per_warp * warps;
  // 16-byte loads of the halves when every half is 16-byte aligned (the base is).
  a.vec = (S * int(sizeof(Tin))) % 16 == 0;
  // With fewer tasks than resident warps (a decode step) each task gets a pair of warps:
  // the two halves run side by side.  (Occupancy is the same for both kernels.)
  const void* fn1 = kmax <= 128 ? reinterpret_cast<const void*>(&select_kernel<Tin, 4, false>)
                                : reinterpret_cast<const void*>(&select_kernel<Tin, 32, false>);
  const void* fn2 = kmax <= 128 ? reinterpret_cast<const void*>(&select_kernel<Tin, 4, true>)
                                : reinterpret_cast<const void*>(&select_kernel<Tin, 32, true>);
  const void* fn = fn1;
  if (cudaFuncSetAttribute(fn1, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)) != cudaSuccess ||
      cudaFuncSetAttribute(fn2, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)) != cudaSuccess)
    return SDM_ECUDA;
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, warps * 32, smem) != cudaSuccess)
    return SDM_ECUDA;
  // About 64 waves of blocks: the last wave is short, and a block's staircase set-up is
  // spread over several tasks per warp.
  const long long tasks = items * 2;
  const long long resident = (long long)sms * (per_sm > 0 ? per_sm : 1) * warps;
  const bool pair = tasks < resident && warps % 2 == 0;
  if (pair) fn = fn2;
  const int units = pair ? warps / 2 : warps;
  long long tpw = tasks / (resident * 64);
  tpw = tpw < 1 ? 1 : (tpw > 64 ? 64 : tpw);
  a.tpw = int(tpw);
  const long long blocks = (tasks + units * tpw - 1) / (units * tpw);
  if (blocks > 0x7FFFFFFFLL) return SDM_EUNSUPPORTED;
  void* args[] = {&a};
  if (cudaLaunchKernel(fn, dim3(unsigned(blocks)), dim3(warps * 32), args, smem, s) != cudaSuccess)
    return SDM_ECUDA;
  return last_launch_status();
}

// Both staircases into out: the write staircase, then the read staircase (one block).
__global__ void stair_table_kernel(uint32_t* out, int W, int R, int S) {
  __shared__ int tmp[32];
  build_stair(out, W, min(W, S), tmp);
  build_stair(out + stair_count(W, min(W, S)), R, min(R, S), tmp);
}

}  // namespace
}  // namespace sdm
