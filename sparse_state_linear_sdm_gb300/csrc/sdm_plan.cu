// Planning pass of the sparse gated-delta scan (Sparse Delta Memory technical summary,
// gist.science/it/paper/2607.07386, "Meccanismo Core" items 3 and 4).
//
// Time-parallel: one block per (b, h, chunk of tokens).  For every token and every
// selected slot it finds whether a token at most `pd` steps earlier (or the same token,
// for a read slot) wrote that slot, and where in that token's write set, so that the
// sequential scan can take the freshly written row from shared memory instead of HBM.
// It also forms both softmaxes (write weights k_t^(i), read weights) and packs slots,
// weights, sources, alpha, beta and v into one 16-byte-aligned record per token (layout
// in sdm_internal.cuh).
//
// Lookups go through an open-addressing table of the chunk's write slots (at most half
// full) behind a 32K-bit filter: a slot whose filter bit is clear was written by no token
// of the chunk, which is the answer for the large majority of slots.
#include "sdm_internal.cuh"

namespace sdm {
namespace {

constexpr int kPlanThreads = 256;
constexpr int kFilterWords = 1024;  // 32,768 filter bits
constexpr unsigned long long kEmpty = ~0ull;

__device__ __forceinline__ uint32_t slot_hash(int32_t x, int log2cap) {
  return (uint32_t(x) * 0x9E3779B1u) >> (32 - log2cap);
}
__device__ __forceinline__ uint32_t filter_bit(int32_t x) {
  return (uint32_t(x) * 0x85EBCA6Bu) >> 17;  // 15 bits
}

template <typename Tv>
__device__ __forceinline__ float load_v(const Tv* p, size_t i);
template <>
__device__ __forceinline__ float load_v<float>(const float* p, size_t i) {
  return p[i];
}
template <>
__device__ __forceinline__ float load_v<uint16_t>(const uint16_t* p, size_t i) {
  return __uint_as_float(uint32_t(p[i]) << 16);
}

struct PlanArgs {
  const int32_t* idx_w;
  const float* sc_w;
  const int32_t* idx_r;
  const float* sc_r;
  const void* v;
  const float* alpha;
  const float* beta;
  int T;        // tokens of the window
  int T_total;  // tokens per sequence in the per-token input arrays
  int t_off;    // first token of the window
  long long N;
  int d_v, W, R, pd, tc;
  int log2cap;  // hash table of 2^log2cap entries, at least twice the entries inserted
  RecLayout L;
  unsigned char* rec;
  int* dev_err;
};

// Shared memory of one planning block: hash table, filter, then the chunk's write slots
// (tokens [t0 - pd, t1)) and read slots (tokens [t0, t1)).
__host__ __device__ inline size_t plan_smem_bytes(int log2cap, int tc, int pd, int W, int R) {
  return (size_t(8) << log2cap) + size_t(kFilterWords) * 4 + size_t(tc + pd) * W * 4 +
         size_t(tc) * R * 4;
}

template <typename Tv>
__global__ void __launch_bounds__(kPlanThreads) plan_kernel(PlanArgs a) {
  // Table entry: slot << 32 | (token - tl) << 16 | position in that token's write set.
  extern __shared__ unsigned long long table[];
  const int tid = threadIdx.x;
  const int bh = blockIdx.y;
  const int t0 = blockIdx.x * a.tc;
  const int t1 = min(a.T, t0 + a.tc);
  const int tl = max(0, t0 - a.pd);
  const int W = a.W, R = a.R, WR = W + R;
  const size_t tok0 = size_t(bh) * a.T_total + a.t_off;  // inputs: token (bh, t_off + u)
  const size_t rec0 = size_t(bh) * a.T;                   // records: (bh, u) of the window
  const int cap = 1 << a.log2cap, mask = cap - 1;
  uint32_t* filter = reinterpret_cast<uint32_t*>(table + cap);
  int32_t* iw = reinterpret_cast<int32_t*>(filter + kFilterWords);  // [(t1 - tl) * W]
  int32_t* ir = iw + (a.tc + a.pd) * W;                               // [(t1 - t0) * R]

  // Stage the slot lists with independent loads (one memory latency, not one per use).
  {
    const int nw = (t1 - tl) * W, nr = (t1 - t0) * R;
    const int32_t* gw = a.idx_w + (tok0 + tl) * W;
    const int32_t* gr = a.idx_r + (tok0 + t0) * R;
#pragma unroll 8
    for (int i = tid; i < nw; i += kPlanThreads) iw[i] = gw[i];
#pragma unroll 8
    for (int i = tid; i < nr; i += kPlanThreads) ir[i] = gr[i];
  }
  for (int i = tid; i < cap; i += kPlanThreads) table[i] = kEmpty;
  for (int i = tid; i < kFilterWords; i += kPlanThreads) filter[i] = 0u;
  __syncthreads();
  const int nins = (t1 - tl) * W;
  for (int k = tid; k < nins; k += kPlanThreads) {
    const int32_t x = iw[k];
    if (x < 0 || x >= a.N) continue;
    const int tt = k / W, pos = k - tt * W;
    const unsigned long long e =
        (static_cast<unsigned long long>(uint32_t(x)) << 32) | (uint32_t(tt) << 16) | uint32_t(pos);
    uint32_t h = slot_hash(x, a.log2cap);
    while (atomicCAS(&table[h], kEmpty, e) != kEmpty) h = (h + 1) & mask;
    const uint32_t fb = filter_bit(x);
    atomicOr(&filter[fb >> 5], 1u << (fb & 31));
  }
  __syncthreads();

  int errs = 0;  // SDM_DEV_* bits seen by this thread, reported once at the end
  for (int u = t0; u < t1; ++u) {
    unsigned char* rec = a.rec + (rec0 + u) * size_t(a.L.bytes);
    for (int e = tid; e < WR; e += kPlanThreads) {
      int32_t x = e < W ? iw[(u - tl) * W + e] : ir[(u - t0) * R + (e - W)];
      int code = -1;
      if (x < 0 || x >= a.N) {
        code = -2;
        x = 0;
        errs |= SDM_DEV_INDEX_RANGE;
      } else {
        const uint32_t fb = filter_bit(x);
        if ((filter[fb >> 5] >> (fb & 31)) & 1u) {
          int best_t = -1, best_p = 0;
          for (uint32_t h = slot_hash(x, a.log2cap);; h = (h + 1) & mask) {
            const unsigned long long v = table[h];
            if (v == kEmpty) break;
            if (uint32_t(v >> 32) != uint32_t(x)) continue;
            const int tt = tl + int((v >> 16) & 0xFFFFu), pp = int(v & 0xFFFFu);
            if (e < W && tt == u && pp != e) errs |= SDM_DEV_DUP_WRITE;
            const bool earlier = e < W ? tt < u : tt <= u;
            if (earlier && tt >= u - a.pd && tt > best_t) {
              best_t = tt;
              best_p = pp;
            }
          }
          if (best_t >= 0) code = (u - best_t) * W + best_p;
        }
      }
      reinterpret_cast<int32_t*>(rec)[e] = x;
      reinterpret_cast<int16_t*>(rec + a.L.off_src)[e] = int16_t(code);
    }
  }

  if (errs && a.dev_err) atomicOr(a.dev_err, errs);

  // Weights, gates and v for each token of the chunk: one warp per token.
  const int warp = tid >> 5, lane = tid & 31;
  for (int u = t0 + warp; u < t1; u += kPlanThreads / 32) {
    unsigned char* rec = a.rec + (rec0 + u) * size_t(a.L.bytes);
    float* wts = reinterpret_cast<float*>(rec + a.L.off_wts);
    warp_softmax(a.sc_w + (tok0 + u) * W, W, wts);
    warp_softmax(a.sc_r + (tok0 + u) * R, R, wts + W);
    if (lane == 0) {
      float* ab = reinterpret_cast<float*>(rec + a.L.off_ab);
      ab[0] = a.alpha[tok0 + u];
      ab[1] = a.beta[tok0 + u];
      ab[2] = 0.f;
      ab[3] = 0.f;
    }
    float* vr = reinterpret_cast<float*>(rec + a.L.off_v);
    const Tv* vsrc = static_cast<const Tv*>(a.v) + (tok0 + u) * size_t(a.d_v);
    for (int c = lane; c < a.d_v; c += 32) vr[c] = load_v<Tv>(vsrc, c);
  }
}

}  // namespace

int launch_plan(const int32_t* idx_w, const float* sc_w, const int32_t* idx_r, const float* sc_r,
                const void* v, int v_dt, const float* alpha, const float* beta,
                const TokenWindow& win, long long N, int d_v, int W, int R, int pd, void* rec,
                int* dev_err, cudaStream_t s) {
  const int T = win.Tc, BH = win.BH;
  if (T == 0 || BH == 0) return SDM_OK;
  PlanArgs pa;
  pa.idx_w = idx_w;
  pa.sc_w = sc_w;
  pa.idx_r = idx_r;
  pa.sc_r = sc_r;
  pa.v = v;
  pa.alpha = alpha;
  pa.beta = beta;
  pa.T = T;
  pa.T_total = win.T_total;
  pa.t_off = win.t0;
  pa.N = N;
  pa.d_v = d_v;
  pa.W = W;
  pa.R = R;
  pa.pd = pd;
  // Tokens per block: at most ~2048 inserted write slots, and shared memory within 96 KB
  // (two blocks per SM); the table has at least twice the inserted entries.
  int tc = 2048 / W - pd;
  tc = tc < 1 ? 1 : (tc > 128 ? 128 : tc);
  auto cap_for = [&](int t) {
    int l = 12;
    while ((1LL << l) < 2LL * (t + pd) * W) ++l;
    return l;
  };
  while (tc > 1 && plan_smem_bytes(cap_for(tc), tc, pd, W, R) > 96 * 1024) --tc;
  pa.tc = tc;
  pa.log2cap = cap_for(tc);
  pa.L = rec_layout(W, R, d_v);
  pa.rec = static_cast<unsigned char*>(rec);
  pa.dev_err = dev_err;
  const dim3 grid((T + tc - 1) / tc, BH);
  const int smem = int(plan_smem_bytes(pa.log2cap, tc, pd, W, R));
  const void* fn = v_dt == SDM_BF16 ? reinterpret_cast<const void*>(&plan_kernel<uint16_t>)
                                    : reinterpret_cast<const void*>(&plan_kernel<float>);
  if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
    return SDM_ECUDA;
  void* args[] = {&pa};
  if (cudaLaunchKernel(fn, grid, dim3(kPlanThreads), args, size_t(smem), s) != cudaSuccess)
    return SDM_ECUDA;
  return last_launch_status();
}

}  // namespace sdm
