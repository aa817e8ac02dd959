// One decode token for a batch of sequences in a single kernel (Sparse Delta Memory
// technical summary, gist.science/it/paper/2607.07386, "Meccanismo Core" items 2-4, with
// T = 1): product-key selection, the planning of the token, and the gated delta write and
// read of its rows, with the state resident in HBM.
//
// The three-kernel path (sdm_select, planning, scan) spends most of a decode step in
// launch and dependency latency: three small grids, each waiting for the previous one's
// writes.  Here one block per (b, h) does all of it:
//   1. the selection of (b, h): in 512-thread blocks warps 0-7 take the k' task and warps
//      8-15 the q' task (teams, below); where the teams' buffers do not fit or K > 128,
//      256-thread blocks with the selection kernel's warp pairs.  Written to idx/sc as
//      sdm_select does.
//   2. the planning of the one token: softmax of the selected write and read scores (the
//      same warp routine as the planning kernel), the source of every row (HBM, or the
//      updated row of the token's own write set for a read slot it also writes, found
//      through a small hash of the write slots), and the device error checks.
//   3. the scan of the token by groups of 256 threads, each taking column slices in turn
//      with the scan kernel's thread mapping and arithmetic for a block of that slice:
//      gather, forget gate and delta update, write-back, weighted read (a read slot the
//      token also writes taking the updated row in place) reduced
//      in the same order.  The slice width is the one the scan kernel would use for these
//      sizes (choose_scan_shape), so the read's sum runs in the same order too.
// So every output is bit-identical to the three-kernel path.
#include "sdm_select_impl.cuh"

namespace sdm {
namespace {


struct DecodeArgs {
  SelectArgs sel;  // one token per (b, h): items = B * H, Tc = T_total = 1
  const void* v;
  const float* alpha;
  const float* beta;
  float* M;
  float* o;
  long long N;
  int d_v, W, R, slices;
  int cols;   // columns of d_v per slice (4 .. 64), as the scan kernel's shape
  int bufs;   // row buffers per group of 256 threads (1 or 2)
  size_t sel_smem;  // bytes of the selection's shared memory
  int* dev_err;
  int parts;  // blocks per (b, h): each repeats the selection and takes its share of the slices
  int pair;   // 1: the two blocks of a (b, h) form a cluster, block r selects task r (k', q')
              // with all its threads and the two exchange their slots and scores
};

// The blocks of a cluster meet (every thread of both; their shared memory writes before are
// visible to the other block after).
__device__ __forceinline__ void decode_cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// A word into the other block's shared memory, at the address this block's copy has (made
// visible to the other block by the next cluster barrier).
__device__ __forceinline__ void decode_peer_store(const void* local, uint32_t peer, uint32_t v) {
  uint32_t addr = static_cast<uint32_t>(__cvta_generic_to_shared(local)), remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(addr), "r"(peer));
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(remote), "r"(v) : "memory");
}

// Shared memory of the planning and scan parts for NG groups of 256 threads with NB row
// buffers each.
__host__ __device__ inline size_t decode_scan_smem(int W, int R, int C, int NG, int NB) {
  const int WR = W + R, WRa = (WR + 3) & ~3;
  int P = 64;
  while (P < 2 * W) P <<= 1;
  return size_t(NG) * NB * WR * C * 4 /* rows */ + size_t(NG) * 8 * C * 4 /* reductions */ +
         size_t(WRa) * 4 /* weights */ + size_t(WRa) * 4 /* slots */ +
         size_t((WRa + 7) & ~7) * 2 /* sources */ + size_t(P) * 4 /* write-slot table */;
}

template <typename Tv>
__device__ __forceinline__ float v_at(const Tv* p, size_t i);
template <>
__device__ __forceinline__ float v_at<float>(const float* p, size_t i) {
  return p[i];
}
template <>
__device__ __forceinline__ float v_at<uint16_t>(const uint16_t* p, size_t i) {
  return __uint_as_float(uint32_t(p[i]) << 16);
}

__device__ __forceinline__ void cp16(float* dst, const float* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(static_cast<uint32_t>(
                   __cvta_generic_to_shared(dst))),
               "l"(src)
               : "memory");
}

// ---- latency-oriented selection for one token: a team of warps per task --------------
//
// The selection kernel gives a task one warp (or two), which suits throughput; for a single
// token the task's latency is what counts.  Here a task gets a team of 256 threads (128 per
// half for the inner lists): radix passes over 8-bit digits narrow the candidates (each
// pass: histogram, the bucket holding the k-th key, compaction), and once at most 64 are
// left they are ranked against each other; the selected keys are put in order by rank.
// The keys are the selection kernel's (distinct: value or sum, then index or flat), so the
// top-k sets and their order are unique and the results are bit-identical.

__device__ __forceinline__ void team_bar(int bar, int nth) {
  asm volatile("bar.sync %0, %1;" ::"r"(bar), "r"(nth) : "memory");
}

// How many of a[0..n) are larger than k: four independent counts, so that the loads of a
// step overlap instead of following each other.
template <typename Key>
__device__ __forceinline__ int count_greater(const Key* a, int n, Key k) {
  int c0 = 0, c1 = 0, c2 = 0, c3 = 0, j = 0;
  for (; j + 4 <= n; j += 4) {
    const Key x0 = a[j], x1 = a[j + 1], x2 = a[j + 2], x3 = a[j + 3];
    c0 += x0 > k ? 1 : 0;
    c1 += x1 > k ? 1 : 0;
    c2 += x2 > k ? 1 : 0;
    c3 += x3 > k ? 1 : 0;
  }
  for (; j < n; ++j) c0 += a[j] > k ? 1 : 0;
  return c0 + c1 + c2 + c3;
}

// The `need` largest of the n distinct keys in a[] into sel[0..need), in no order; a and b
// (n entries each) are overwritten.  `bits`: key width (multiple of 8).  hist: 256
// counters, ctr: 4 ints, both team-private.  Team thread t of nth (whole warps), barrier bar.
template <typename Key>
__device__ void team_topk(Key* a, Key* b, int n, int need, int bits, Key* sel, uint32_t* hist,
                          int* ctr, int t, int nth, int bar) {
  int shift = bits - 8, nsel = 0, left = need;
  if (t == 0) ctr[0] = 0;
  // the histogram is cleared here for the first pass and, for each later one, while the
  // previous pass appends (no pass reads it after its bucket search)
  for (int i = t; i < 256; i += nth) hist[i] = 0u;
  team_bar(bar, nth);
  for (;;) {
    if (n <= left) {  // every candidate is in
      for (int i = t; i < n; i += nth) sel[nsel + i] = a[i];
      team_bar(bar, nth);
      return;
    }
    if (n <= 64 || shift < 0) {  // rank the few candidates left
      for (int i = t; i < n; i += nth) {
        const int r = count_greater(a, n, a[i]);
        if (r < left) sel[nsel + r] = a[i];
      }
      team_bar(bar, nth);
      return;
    }
    // Equal digits of a warp are counted with one atomic (few bins take most keys).
    for (int i0 = 0; i0 < n; i0 += nth) {
      const int i = i0 + t;
      const unsigned dg = i < n ? unsigned(a[i] >> shift) & 255u : 256u;
      const unsigned same = __match_any_sync(kFull, dg);
      if (dg < 256u && (threadIdx.x & 31) == __ffs(same) - 1) atomicAdd(&hist[dg], unsigned(__popc(same)));
    }
    team_bar(bar, nth);
    if (t < 32) {  // the bucket of the left-th largest key: lane l owns bins 8l .. 8l+7
      uint32_t own = 0;
#pragma unroll
      for (int d = 0; d < 8; ++d) own += hist[8 * t + d];
      uint32_t suf = own;  // keys in the bins of lanes >= t
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const uint32_t y = __shfl_down_sync(kFull, suf, off);
        if (t + off < 32) suf += y;
      }
      const unsigned ok = __ballot_sync(kFull, suf >= uint32_t(left));
      const int L = 31 - __clz(int(ok));
      if (t == L) {
        uint32_t run = suf - own;
        for (int d = 7; d >= 0; --d) {
          const uint32_t hcount = hist[8 * t + d];
          if (run + hcount >= uint32_t(left)) {
            ctr[1] = 0;
            ctr[2] = 8 * t + d;
            ctr[3] = int(run);
            break;
          }
          run += hcount;
        }
      }
    }
    team_bar(bar, nth);
    const uint32_t bstar = uint32_t(ctr[2]);
    const int above = ctr[3];
    for (int i = t; i < 256; i += nth) hist[i] = 0u;  // for the next pass
    // Appends with one atomic per warp and list (ballot, then each lane's rank in it).
    const unsigned lane = threadIdx.x & 31, below = (1u << lane) - 1u;
    for (int i0 = 0; i0 < n; i0 += nth) {
      const int i = i0 + t;
      Key k = 0;
      uint32_t dg = 0;
      if (i < n) {
        k = a[i];
        dg = unsigned(k >> shift) & 255u;
      }
      const unsigned up = __ballot_sync(kFull, i < n && dg > bstar);
      const unsigned eq = __ballot_sync(kFull, i < n && dg == bstar);
      int base_up = 0, base_eq = 0;
      if (lane == 0) {
        if (up) base_up = atomicAdd(&ctr[0], __popc(up));
        if (eq) base_eq = atomicAdd(&ctr[1], __popc(eq));
      }
      base_up = __shfl_sync(kFull, base_up, 0);
      base_eq = __shfl_sync(kFull, base_eq, 0);
      if ((up >> lane) & 1u) sel[base_up + __popc(up & below)] = k;
      if ((eq >> lane) & 1u) b[base_eq + __popc(eq & below)] = k;
    }
    team_bar(bar, nth);
    nsel += above;
    left -= above;
    n = ctr[1];
    Key* sw = a;
    a = b;
    b = sw;
    shift -= 8;
  }
}

// Both staircases {(p, q): p, q < kin, (p+1)(q+1) <= K} as p << 16 | q, row by row, with
// every thread of the block: warp 0 (W) and warp 1 (R) form the rows' start offsets, then
// each entry finds its row by binary search.  rs: (kin_w + 1) + (kin_r + 1) ints of scratch.
__device__ void build_stairs_parallel(uint32_t* st_w, uint32_t* st_r, int W, int R, int S,
                                      int* rs, int nt) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int kw = min(W, S), kr = min(R, S);
  int* rs_w = rs;
  int* rs_r = rs + kw + 1;
  if (warp < 2) {
    const int K = warp ? R : W, kin = warp ? kr : kw;
    int* r = warp ? rs_r : rs_w;
    const int per = (kin + 31) / 32;
    const int p0 = min(kin, lane * per), p1 = min(kin, p0 + per);
    int mine = 0;
    for (int p = p0; p < p1; ++p) mine += min(kin, K / (p + 1));
    int incl = mine;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(kFull, incl, off);
      if (lane >= off) incl += y;
    }
    int off = incl - mine;
    for (int p = p0; p < p1; ++p) {
      r[p] = off;
      off += min(kin, K / (p + 1));
    }
    if (lane == 31) r[kin] = incl;
  }
  __syncthreads();
  for (int which = 0; which < 2; ++which) {
    const int kin = which ? kr : kw;
    const int* r = which ? rs_r : rs_w;
    uint32_t* st = which ? st_r : st_w;
    const int cnt = r[kin];
    for (int c = tid; c < cnt; c += nt) {
      int lo = 0, hi = kin - 1;  // the last row starting at or before c
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (r[mid] <= c) lo = mid; else hi = mid - 1;
      }
      st[c] = (uint32_t(lo) << 16) | uint32_t(c - r[lo]);
    }
  }
  __syncthreads();
}

// Shared memory of one team.
struct TeamMem {
  unsigned char* A;  // inner keys of both halves, then the staircase keys
  unsigned char* B;  // their scratch
  unsigned char* isel;  // inner selections [2][kin_max] inner keys
  uint64_t* osel;       // outer selection [kpad]
  uint64_t* oout;       // outer selection in order [kpad]
  uint32_t* hist;       // [2][256]
  int* ctr;             // [2][4], then a flag
  float* aval;          // [kin_max] x 2 lists
  float* bval;
  int32_t* aidx;
  int32_t* bidx;
  int32_t* ridx;        // the task's result: slots [kpad]
  float* rsc;           // and scores [kpad]
};

__host__ __device__ inline size_t team_buf_bytes(int S, int cnt_max, int ikb) {
  size_t x = size_t(2) * S * ikb;
  if (size_t(cnt_max) * 8 > x) x = size_t(cnt_max) * 8;
  return (x + 15) / 16 * 16;
}
__host__ __device__ inline size_t team_mem_bytes(int S, int kin_max, int kpad, int cnt_max, int ikb) {
  const size_t buf = team_buf_bytes(S, cnt_max, ikb);
  return 2 * buf + (size_t(2) * kin_max * ikb + 15) / 16 * 16 + size_t(2) * kpad * 8 +
         size_t(512) * 4 + 48 + size_t(4) * kin_max * 4 + size_t(2) * kpad * 4;
}

__device__ __forceinline__ TeamMem team_mem(unsigned char* base, int S, int kin_max, int kpad,
                                            int cnt_max, int ikb) {
  TeamMem m;
  const size_t buf = team_buf_bytes(S, cnt_max, ikb);
  m.A = base;
  m.B = base + buf;
  m.isel = base + 2 * buf;
  unsigned char* q = m.isel + (size_t(2) * kin_max * ikb + 15) / 16 * 16;
  m.osel = reinterpret_cast<uint64_t*>(q);
  m.oout = m.osel + kpad;
  m.hist = reinterpret_cast<uint32_t*>(m.oout + kpad);
  m.ctr = reinterpret_cast<int*>(m.hist + 512);
  m.aval = reinterpret_cast<float*>(reinterpret_cast<unsigned char*>(m.ctr) + 48);
  m.bval = m.aval + kin_max;
  m.aidx = reinterpret_cast<int32_t*>(m.bval + kin_max);
  m.bidx = m.aidx + kin_max;
  m.ridx = m.bidx + kin_max;
  m.rsc = reinterpret_cast<float*>(m.ridx + kpad);
  return m;
}

// Task `which` (0: k' / top-W, 1: q' / top-R) of token `item` by a team of TT threads
// (team thread t); barriers bar0 (the team), bar0 + 1 and bar0 + 2 (its two halves).
// peer >= 0: the slots and scores are also stored into the cluster block `peer`'s copy of
// push_idx / push_sc.
template <typename Tin, int EMAX, int TT>
__device__ void team_select(const SelectArgs& a, long long item, int which, const uint32_t* stair,
                            const TeamMem& m, int t, int bar0, bool write_out = true, int peer = -1,
                            int32_t* push_idx = nullptr, float* push_sc = nullptr) {
  using IKey = typename InnerKeyOf<Tin>::type;
  constexpr int IBITS = sizeof(Tin) == 2 ? 32 : 48;
  const int S = a.S, K = which ? a.R : a.W, kin = min(K, S);
  const int cnt = which ? a.cnt_r : a.cnt_w;
  const Tin* halves = static_cast<const Tin*>(which ? a.qp : a.kp) + item * 2 * S;

  constexpr int HT = TT / 2;  // threads per half
  // ---- inner: half h by threads HT*h .. HT*h + HT-1 ----
  {
    const int h = t / HT, ht = t % HT, hb = bar0 + 1 + h;
    IKey* A = reinterpret_cast<IKey*>(m.A) + size_t(h) * S;
    IKey* Bk = reinterpret_cast<IKey*>(m.B) + size_t(h) * S;
    IKey* sel = reinterpret_cast<IKey*>(m.isel) + size_t(h) * a.kin_max;
    const Tin* src = halves + size_t(h) * S;
    constexpr int EPV = 16 / int(sizeof(Tin));
    if (a.vec) {  // 16-byte loads, up to four per thread issued before any is used
      const uint4* src4 = reinterpret_cast<const uint4*>(src);
      const int nvec = S / EPV;
      for (int c0 = ht; c0 < nvec; c0 += HT * 4) {
        uint4 q[4];
#pragma unroll
        for (int u = 0; u < 4; ++u)
          q[u] = c0 + HT * u < nvec ? __ldg(src4 + c0 + HT * u) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int c = c0 + HT * u;
          if (c >= nvec) break;
          float f[EPV];
          unpack16<Tin>(q[u], f);
#pragma unroll
          for (int i = 0; i < EPV; ++i)
            A[c * EPV + i] = inner_key_f(f[i], c * EPV + i, static_cast<IKey*>(nullptr));
        }
      }
    } else {
      for (int j0 = ht; j0 < S; j0 += HT * 8) {
        Tin q[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) q[u] = j0 + HT * u < S ? src[j0 + HT * u] : Tin(0);
#pragma unroll
        for (int u = 0; u < 8; ++u)
          if (j0 + HT * u < S) A[j0 + HT * u] = inner_key(q[u], j0 + HT * u);
      }
    }
    team_bar(hb, HT);
    team_topk<IKey>(A, Bk, S, kin, IBITS, sel, m.hist + 256 * h, m.ctr + 4 * h, ht, HT, hb);
    float* dv = h ? m.bval : m.aval;
    int32_t* di = h ? m.bidx : m.aidx;
    for (int i = ht; i < kin; i += HT) {
      const IKey k = sel[i];
      const int r = count_greater(sel, kin, k);
      dv[r] = inner_value(k);
      di[r] = min(int(0xFFFFu - uint32_t(k & 0xFFFFu)), S - 1);
    }
  }
  team_bar(bar0, TT);

  // ---- outer: top-K of the staircase pairs ----
  const float* aval = m.aval;
  const float* bval = m.bval;
  const int32_t* aidx = m.aidx;
  const int32_t* bidx = m.bidx;
  auto pair_key = [&](int p, int q) -> uint64_t {
    const float sum = __fadd_rn(aval[p], bval[q]);
    const uint32_t flat = uint32_t(aidx[p]) * uint32_t(S) + uint32_t(bidx[q]);
    return (uint64_t(ord_key(sum)) << 32) | uint64_t(0xFFFFFFFFu - flat);
  };
  uint64_t* OA = reinterpret_cast<uint64_t*>(m.A);
  uint64_t* OB = reinterpret_cast<uint64_t*>(m.B);
  for (int c = t; c < cnt; c += TT) {
    const uint32_t pq = stair[c];
    OA[c] = pair_key(int(pq >> 16), int(pq & 0xFFFFu));
  }
  team_bar(bar0, TT);
  team_topk<uint64_t>(OA, OB, cnt, K, 64, m.osel, m.hist, m.ctr, t, TT, bar0);
  for (int i = t; i < K; i += TT) {
    const uint64_t k = m.osel[i];
    m.oout[count_greater(m.osel, K, k)] = k;
  }
  if (t == 0) m.ctr[8] = 0;
  team_bar(bar0, TT);
  // Pairs right of the staircase that could still beat the K-th key.
  const uint64_t kth = m.oout[K - 1];
  const uint32_t kth_sum = uint32_t(kth >> 32);
  bool beyond = false;
  for (int p = t; p < kin; p += TT) {
    for (int q = min(kin, K / (p + 1)); q < kin; ++q) {
      const uint64_t k = pair_key(p, q);
      if (uint32_t(k >> 32) < kth_sum) break;  // sums only fall along a row
      if (k > kth) beyond = true;
    }
  }
  if (beyond) m.ctr[8] = 1;
  team_bar(bar0, TT);
  if (m.ctr[8]) {  // rare: redo over every grid pair that can reach the K-th key
    if (t < 32) {
      outer_full_grid(aval, bval, aidx, bidx, S, kin, K, kth, m.oout, a.kpad, m.hist);
      sort_desc_upto<uint64_t, EMAX>(m.oout, K);
    }
    team_bar(bar0, TT);
  }
  int32_t* oi = (which ? a.idx_r : a.idx_w) + item * K;
  float* os = (which ? a.sc_r : a.sc_w) + item * K;
  // the other block has started (its arrive at the kernel's start) before anything is stored
  // into its shared memory
  if (peer >= 0) asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
  for (int r = t; r < K; r += TT) {
    const uint64_t k = m.oout[r];
    const int32_t slot = int32_t(0xFFFFFFFFu - uint32_t(k & 0xFFFFFFFFu));
    const float sc = ord_decode(uint32_t(k >> 32));
    if (write_out) {
      oi[r] = slot;
      os[r] = sc;
    }
    m.ridx[r] = slot;
    m.rsc[r] = sc;
    if (peer >= 0) {
      decode_peer_store(push_idx + r, uint32_t(peer), uint32_t(slot));
      decode_peer_store(push_sc + r, uint32_t(peer), __float_as_uint(sc));
    }
  }
}

template <typename Tin, typename Tv, int EMAX, bool TEAM>
__global__ void __launch_bounds__(TEAM ? 512 : 256, 1) decode_kernel(DecodeArgs d) {
  constexpr int NT = TEAM ? 512 : 256;  // threads of the block
  constexpr int NG = NT / 256;          // groups of 256 threads scanning slices side by side
  extern __shared__ __align__(16) unsigned char smem[];
  const SelectArgs& a = d.sel;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // d.parts blocks per (b, h) (the team path only): each selects and plans the token, part 0
  // writes the selection's outputs, and part p scans slices p*NG .. p*NG+NG-1, then every
  // parts*NG-th one after them.
  const int bh = blockIdx.x / d.parts, part = blockIdx.x - bh * d.parts;
  const int C = d.cols, LPR = C / 4, RPP = 256 / LPR;
  const int W = d.W, R = d.R, WR = W + R, d_v = d.d_v;
  // cluster pair: this block has started (waited on before the other block stores into it)
  if (TEAM && d.pair) asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
  const float alpha = d.alpha[bh], beta = d.beta[bh];

  // ---- 1. selection of token (bh, 0) -------------------------------------------------
  const int32_t* gw = a.idx_w + size_t(bh) * W;
  const int32_t* gr = a.idx_r + size_t(bh) * R;
  const float* sw = a.sc_w + size_t(bh) * W;
  const float* sr = a.sc_r + size_t(bh) * R;
  unsigned char* sbase = smem;
  if (TEAM) {  // warps 0-7: the k' task, warps 8-15: the q' task
    constexpr int ikb = int(sizeof(typename InnerKeyOf<Tin>::type));
    uint32_t* stair_w = reinterpret_cast<uint32_t*>(smem);
    uint32_t* stair_r = stair_w + a.cnt_w;
    unsigned char* tbase = smem + (size_t(a.cnt_w + a.cnt_r) * 4 + 15) / 16 * 16;
    const int cmax = max(a.cnt_w, a.cnt_r);
    const size_t tsize = (team_mem_bytes(a.S, a.kin_max, a.kpad, cmax, ikb) + 15) / 16 * 16;
    const TeamMem m0 = team_mem(tbase, a.S, a.kin_max, a.kpad, cmax, ikb);
    const TeamMem m1 = team_mem(tbase + tsize, a.S, a.kin_max, a.kpad, cmax, ikb);
    if (a.stair_g) {  // prebuilt by the caller (sdm_decode_table)
      stair_w = const_cast<uint32_t*>(a.stair_g);
      stair_r = stair_w + a.cnt_w;
    } else {  // team 0's histograms are free until its selection starts: scratch for them
      build_stairs_parallel(stair_w, stair_r, a.W, a.R, a.S, reinterpret_cast<int*>(m0.hist), NT);
    }
    if (d.pair) {
      // Block `part` of the cluster takes task `part` (0: k', 1: q') with every thread and
      // stores its slots and scores into its own m0 and the other block's m1 (which the
      // selection does not use); one cluster barrier then makes both blocks' stores visible,
      // and no block touches the other's shared memory after it.
      team_select<Tin, EMAX, NT>(a, bh, part, part ? stair_r : stair_w, m0, tid, 1, true,
                                 part ^ 1, m1.ridx, m1.rsc);
      decode_cluster_sync();
      gw = part ? m1.ridx : m0.ridx;
      sw = part ? m1.rsc : m0.rsc;
      gr = part ? m0.ridx : m1.ridx;
      sr = part ? m0.rsc : m1.rsc;
    } else {
      const int team = warp >> 3;
      team_select<Tin, EMAX, 256>(a, bh, team, team ? stair_r : stair_w, team ? m1 : m0,
                                  tid & 255, 1 + 3 * team, part == 0);
      // the slots and scores stay in shared memory; the scan's buffers follow them
      gw = m0.ridx;
      sw = m0.rsc;
      gr = m1.ridx;
      sr = m1.rsc;
    }
    sbase = smem + d.sel_smem;
  } else {  // the selection kernel's pair mode: warps 0-1 the k' task, 2-3 the q' task
    const SelectSmem m = select_smem(a, smem);
    if (!a.stair_g) select_build_stairs(a, m);
    if (warp < 4) {
      const long long task = 2LL * bh + (warp >> 1);
      select_tasks<Tin, EMAX, true>(a, m, task, task + 1);
    }
  }
  __syncthreads();  // the token's slots and scores are written

  // ---- 2. planning of the token -----------------------------------------------------
  const int WRa = (WR + 3) & ~3;
  float* rows = reinterpret_cast<float*>(sbase);                  // [NG][bufs][WR][C]
  float* red = rows + size_t(NG) * d.bufs * WR * C;               // [NG][8][C]
  float* wts = red + NG * 8 * C;                                  // [WRa]
  int32_t* idx = reinterpret_cast<int32_t*>(wts + WRa);           // [WRa]
  int16_t* src = reinterpret_cast<int16_t*>(idx + WRa);           // [WRa]
  int* table = reinterpret_cast<int*>(src + ((WRa + 7) & ~7));    // [P] write positions by slot
  int lg = 6;
  while ((1 << lg) < 2 * W) ++lg;
  const int P = 1 << lg;
  for (int i = tid; i < P; i += NT) table[i] = -1;
  for (int e = tid; e < WR; e += NT) idx[e] = e < W ? gw[e] : gr[e - W];
  if (warp == 0) warp_softmax(sw, W, wts);
  if (warp == 1) warp_softmax(sr, R, wts + W);
  __syncthreads();
  // Write slots into an open-addressing table (a slot met twice: a duplicate write).
  int errs = 0;
  auto slot_hash = [&](int32_t x) { return (uint32_t(x) * 0x9E3779B1u) >> (32 - lg); };
  for (int e = tid; e < W; e += NT) {
    const int32_t x = idx[e];
    if (x < 0 || x >= d.N) continue;
    for (uint32_t h = slot_hash(x);; h = (h + 1) & uint32_t(P - 1)) {
      const int prev = atomicCAS(&table[h], -1, e);
      if (prev == -1) break;
      if (idx[prev] == x) {
        errs |= SDM_DEV_DUP_WRITE;
        break;
      }
    }
  }
  __syncthreads();
  for (int e = tid; e < WR; e += NT) {
    const int32_t x = idx[e];
    int code = -1;
    if (x < 0 || x >= d.N) {
      code = -2;
      errs |= SDM_DEV_INDEX_RANGE;
    } else if (e >= W) {  // a read of a row this token writes: the updated row
      for (uint32_t h = slot_hash(x);; h = (h + 1) & uint32_t(P - 1)) {
        const int p = table[h];
        if (p == -1) break;
        if (idx[p] == x) {
          code = p;
          break;
        }
      }
    }
    src[e] = int16_t(code);
  }
  if (errs && d.dev_err) atomicOr(d.dev_err, errs);
  __syncthreads();

  // ---- 3. the token's scan: group gi of 256 threads takes slices gi, gi+NG, ... ---------
  // Each slice with the scan kernel's thread mapping for a block of that slice; with two
  // row buffers per group the next slice's rows are gathered while this one is computed.
  const int gi = tid >> 8, lt = tid & 255, lw = lt >> 5, gbar = 7 + gi;
  const int NB = d.bufs;  // row buffers per group (1 or 2)
  float* redg = red + gi * 8 * C;
  const int c4 = lt % LPR;
  float* Mbh = d.M + size_t(bh) * size_t(d.N) * d_v;
  auto gather = [&](int sl, float* rg) {
    const float* Mc = Mbh + sl * C;
    for (int e = lt / LPR; e < WR; e += RPP)
      if (src[e] == -1) cp16(rg + e * C + 4 * c4, Mc + size_t(idx[e]) * d_v + 4 * c4);
    asm volatile("cp.async.commit_group;" ::: "memory");
  };
  const int sl0 = part * NG + gi, sstep = d.parts * NG;
  if (sl0 < d.slices) gather(sl0, rows + size_t(gi * NB) * WR * C);
  for (int sl = sl0, k = 0; sl < d.slices; sl += sstep, ++k) {
    const int c0 = sl * C;
    float* Mc = Mbh + c0;
    float* rg = rows + size_t(gi * NB + (k % NB)) * WR * C;
    const bool ahead = NB > 1 && sl + sstep < d.slices;
    if (ahead) gather(sl + sstep, rows + size_t(gi * NB + ((k + 1) % NB)) * WR * C);
    if (ahead)
      asm volatile("cp.async.wait_group 1;" ::: "memory");
    else
      asm volatile("cp.async.wait_group 0;" ::: "memory");
    const Tv* vsrc = static_cast<const Tv*>(d.v) + size_t(bh) * d_v + c0 + 4 * c4;
    const float4 vv = make_float4(v_at<Tv>(vsrc, 0), v_at<Tv>(vsrc, 1), v_at<Tv>(vsrc, 2),
                                  v_at<Tv>(vsrc, 3));
    team_bar(gbar, 256);
    // Forget gate and delta update of the W write rows (in shared memory and in HBM).
    for (int e = lt / LPR; e < W; e += RPP) {
      if (src[e] == -2) continue;
      float4* cell = reinterpret_cast<float4*>(rg + e * C) + c4;
      const float4 m = *cell;
      const float kb = beta * wts[e];
      float4 r;
      float mt_;
      mt_ = alpha * m.x; r.x = fmaf(kb, vv.x - mt_, mt_);
      mt_ = alpha * m.y; r.y = fmaf(kb, vv.y - mt_, mt_);
      mt_ = alpha * m.z; r.z = fmaf(kb, vv.z - mt_, mt_);
      mt_ = alpha * m.w; r.w = fmaf(kb, vv.w - mt_, mt_);
      *cell = r;
      *(reinterpret_cast<float4*>(Mc + size_t(idx[e]) * d_v) + c4) = r;
    }
    team_bar(gbar, 256);
    // Weighted read of the R read rows (after the write), in the scan kernel's order; a read
    // of a row this token also writes takes the updated row where the write left it.
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int e = lt / LPR; e < R; e += RPP) {
      const int code = src[W + e];
      if (code == -2) continue;
      const float r = wts[W + e];
      const int row = code >= 0 && code < W ? code : W + e;
      const float4 m = reinterpret_cast<const float4*>(rg + row * C)[c4];
      acc.x = fmaf(r, m.x, acc.x);
      acc.y = fmaf(r, m.y, acc.y);
      acc.z = fmaf(r, m.z, acc.z);
      acc.w = fmaf(r, m.w, acc.w);
    }
    for (int off = LPR; off < 32; off <<= 1) {
      acc.x += __shfl_xor_sync(0xFFFFFFFFu, acc.x, off);
      acc.y += __shfl_xor_sync(0xFFFFFFFFu, acc.y, off);
      acc.z += __shfl_xor_sync(0xFFFFFFFFu, acc.z, off);
      acc.w += __shfl_xor_sync(0xFFFFFFFFu, acc.w, off);
    }
    if (lane < LPR) reinterpret_cast<float4*>(redg + lw * C)[lane] = acc;
    team_bar(gbar, 256);
    if (lt < LPR) {
      float4 sum = reinterpret_cast<const float4*>(redg)[lt];
#pragma unroll
      for (int w = 1; w < 8; ++w) {
        const float4 t = reinterpret_cast<const float4*>(redg + w * C)[lt];
        sum = make_float4(sum.x + t.x, sum.y + t.y, sum.z + t.z, sum.w + t.w);
      }
      *(reinterpret_cast<float4*>(d.o + size_t(bh) * d_v + c0) + lt) = sum;
    }
    if (NB == 1 && sl + sstep < d.slices) {
      team_bar(gbar, 256);  // every read of this slice's rows is done
      gather(sl + sstep, rg);
    } else if (NB > 1) {
      team_bar(gbar, 256);  // the buffer is gathered into again two slices later
    }
  }
}

// Launch shape of the decode kernel: slice width (the scan kernel's), selection variant
// (teams of 8 warps in 512-thread blocks, or warp pairs in 256-thread blocks), shared memory.
template <typename Tin>
int decode_shape(int BH, int S, int d_v, int W, int R, SelectArgs* sel, int* cols, int* bufs,
                 size_t* smem, size_t* sel_smem, bool* team) {
  ScanShape shape;
  const int st = choose_scan_shape(BH, d_v, W, R, 0, 0, &shape);
  if (st != SDM_OK) return st;
  if (shape.cols < 4 || shape.cols > 64 || d_v % shape.cols != 0) return SDM_EUNSUPPORTED;
  size_t stair_bytes = 0, per_warp = 0;
  select_args<Tin>(nullptr, nullptr, whole_sequences(BH, 1), S, W, R, nullptr, nullptr, nullptr,
                   nullptr, sel, &stair_bytes, &per_warp);
  sel->warps = 4;
  *cols = shape.cols;
  int dev = 0, max_smem = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
    return SDM_ECUDA;
  const size_t cap = size_t(max_smem);
  const int ikb = int(sizeof(typename InnerKeyOf<Tin>::type));
  const size_t team_smem =
      stair_bytes + 2 * ((team_mem_bytes(S, sel->kin_max, sel->kpad, max(sel->cnt_w, sel->cnt_r),
                                         ikb) + 15) / 16 * 16);
  const int slices = d_v / shape.cols;
  // Two row buffers per group where there are slices to prefetch and they fit.
  *bufs = slices > 2 && team_smem + decode_scan_smem(W, R, shape.cols, 2, 2) <= cap ? 2 : 1;
  const size_t team_total = team_smem + decode_scan_smem(W, R, shape.cols, 2, *bufs);
  *team = W <= 128 && R <= 128 && team_total <= cap;
  if (*team) {
    *sel_smem = team_smem;
    *smem = team_total;  // the scan's buffers follow the team selections
  } else {
    *bufs = 1;
    *sel_smem = stair_bytes + 4 * per_warp;
    const size_t sc = decode_scan_smem(W, R, shape.cols, 1, 1);
    *smem = *sel_smem > sc ? *sel_smem : sc;
  }
  return *smem > cap ? SDM_EUNSUPPORTED : SDM_OK;
}

template <typename Tin>
int launch_decode_t(const void* kp, const void* qp, const void* v, int v_dt, const float* alpha,
                    const float* beta, float* M, int BH, int S, int d_v, int W, int R,
                    int32_t* idx_w, float* sc_w, int32_t* idx_r, float* sc_r, float* o,
                    int* dev_err, cudaStream_t s, const uint32_t* stairs) {
  DecodeArgs dargs;
  int cols = 0, bufs = 1;
  size_t smem = 0;
  bool team = false;
  const int st = decode_shape<Tin>(BH, S, d_v, W, R, &dargs.sel, &cols, &bufs, &smem,
                                   &dargs.sel_smem, &team);
  if (st != SDM_OK) return st;
  dargs.sel.kp = kp;
  dargs.sel.qp = qp;
  dargs.sel.idx_w = idx_w;
  dargs.sel.sc_w = sc_w;
  dargs.sel.idx_r = idx_r;
  dargs.sel.sc_r = sc_r;
  dargs.sel.stair_g = stairs;
  dargs.v = v;
  dargs.alpha = alpha;
  dargs.beta = beta;
  dargs.M = M;
  dargs.o = o;
  dargs.N = (long long)S * S;
  dargs.d_v = d_v;
  dargs.W = W;
  dargs.R = R;
  dargs.cols = cols;
  dargs.slices = d_v / cols;
  dargs.bufs = bufs;
  dargs.dev_err = dev_err;
  // Two blocks per (b, h) when the slices take more than one round of the block's groups and
  // both blocks still find an SM of their own: the selection is repeated, the rounds halve.
  int sms = 0, dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return SDM_ECUDA;
  dargs.pair = team && 2LL * BH <= sms ? 1 : 0;
  dargs.parts = dargs.pair || (team && dargs.slices > 2 && 2LL * BH <= sms) ? 2 : 1;
  const bool big = W > 128 || R > 128;
  const void* fn;
  if (v_dt == SDM_BF16)
    fn = big    ? reinterpret_cast<const void*>(&decode_kernel<Tin, uint16_t, 32, false>)
         : team ? reinterpret_cast<const void*>(&decode_kernel<Tin, uint16_t, 4, true>)
                : reinterpret_cast<const void*>(&decode_kernel<Tin, uint16_t, 4, false>);
  else
    fn = big    ? reinterpret_cast<const void*>(&decode_kernel<Tin, float, 32, false>)
         : team ? reinterpret_cast<const void*>(&decode_kernel<Tin, float, 4, true>)
                : reinterpret_cast<const void*>(&decode_kernel<Tin, float, 4, false>);
  if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)) !=
      cudaSuccess)
    return SDM_ECUDA;
  void* args[] = {&dargs};
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(BH * dargs.parts));
  cfg.blockDim = dim3(team ? 512 : 256);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = unsigned(dargs.pair ? 2 : 1);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelExC(&cfg, fn, args) != cudaSuccess) return SDM_ECUDA;
  return last_launch_status();
}

}  // namespace

int launch_decode(const void* kp, const void* qp, int in_dt, const void* v, int v_dt,
                  const float* alpha, const float* beta, float* M, int BH, int S, int d_v, int W,
                  int R, int32_t* idx_w, float* sc_w, int32_t* idx_r, float* sc_r, float* o,
                  int* dev_err, cudaStream_t s, const uint32_t* stairs) {
  if (BH == 0) return SDM_OK;
  return in_dt == SDM_BF16
             ? launch_decode_t<uint16_t>(kp, qp, v, v_dt, alpha, beta, M, BH, S, d_v, W, R, idx_w,
                                         sc_w, idx_r, sc_r, o, dev_err, s, stairs)
             : launch_decode_t<float>(kp, qp, v, v_dt, alpha, beta, M, BH, S, d_v, W, R, idx_w,
                                      sc_w, idx_r, sc_r, o, dev_err, s, stairs);
}

int decode_supported(int in_dt, int BH, int S, int d_v, int W, int R) {
  SelectArgs sel;
  int cols = 0, bufs = 1;
  size_t smem = 0, sel_smem = 0;
  bool team = false;
  return in_dt == SDM_BF16 ? decode_shape<uint16_t>(BH, S, d_v, W, R, &sel, &cols, &bufs, &smem,
                                                    &sel_smem, &team)
                           : decode_shape<float>(BH, S, d_v, W, R, &sel, &cols, &bufs, &smem,
                                                 &sel_smem, &team);
}

}  // namespace sdm
