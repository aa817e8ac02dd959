// Planning pass of the sparse gated-delta scan (Sparse Delta Memory technical summary,
// gist.science/it/paper/2607.07386, "Meccanismo Core" items 3 and 4).
//
// Time-parallel: one warp per token.  For every selected slot of the token it finds whether
// a token at most `pd` steps earlier (or the same token, for a read slot) wrote that slot,
// and where in that token's write set, so that the sequential scan can take the freshly
// written row from shared memory instead of HBM.  It also forms both softmaxes (write
// weights k_t^(i), read weights) and packs slots, weights, sources, alpha, beta and v into
// one 16-byte-aligned record per token (layout in sdm_internal.cuh).
//
// Lookups go through a small open-addressing table per warp (at most half full) holding
// the write sets of the token and of the pd tokens before it in the window; it is rebuilt
// for every token, so no state crosses tokens and every warp is independent.
#include "sdm_internal.cuh"

namespace sdm {
namespace {

constexpr int kPlanMaxWarps = 8;  // warps (tokens) per block, fewer when the tables are large
constexpr unsigned long long kEmpty = ~0ull;

__device__ __forceinline__ uint32_t slot_hash(int32_t x, int log2cap) {
  return (uint32_t(x) * 0x9E3779B1u) >> (32 - log2cap);
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
  int BH;
  long long N;
  int d_v, W, R, pd;
  int log2cap;  // per-warp hash table of 2^log2cap entries, at least twice the entries inserted
  int warps;    // warps per block
  RecLayout L;
  unsigned char* rec;
  int* dev_err;
};

template <typename Tv>
__global__ void __launch_bounds__(kPlanMaxWarps * 32) plan_kernel(PlanArgs a) {
  // Table entry: slot << 32 | (token - first) << 16 | position in that token's write set.
  extern __shared__ unsigned long long tables[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long g = (long long)blockIdx.x * a.warps + warp;  // (bh, u) of the window
  if (g >= (long long)a.BH * a.T) return;
  const int bh = int(g / a.T), u = int(g - (long long)bh * a.T);
  const int W = a.W, R = a.R, WR = W + R;
  const int cap = 1 << a.log2cap, mask = cap - 1;
  unsigned long long* table = tables + size_t(warp) * cap;
  const size_t tok0 = size_t(bh) * a.T_total + a.t_off;  // inputs: token (bh, t_off + u)
  const int first = max(0, u - a.pd);                      // no forwarding from before the window

  // The token's scores first (register softmax below when each lane holds at most four),
  // then the write sets; the loads do not wait for one another.
  const bool reg_softmax = W <= 128 && R <= 128;
  float sw[4], sr[4];
  if (reg_softmax) {
    const float* gsw = a.sc_w + (tok0 + u) * W;
    const float* gsr = a.sc_r + (tok0 + u) * R;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      sw[j] = lane + 32 * j < W ? gsw[lane + 32 * j] : -INFINITY;
      sr[j] = lane + 32 * j < R ? gsr[lane + 32 * j] : -INFINITY;
    }
  }
  for (int i = lane; i < cap; i += 32) table[i] = kEmpty;
  __syncwarp();
  int errs = 0;  // SDM_DEV_* bits seen by this lane, reported once at the end
  const int nins = (u - first + 1) * W;
  const int32_t* gw = a.idx_w + (tok0 + first) * W;
#pragma unroll 4
  for (int k = lane; k < nins; k += 32) {
    const int32_t x = gw[k];
    if (x < 0 || x >= a.N) continue;
    const int tt = k / W, pos = k - tt * W;
    const unsigned long long e =
        (static_cast<unsigned long long>(uint32_t(x)) << 32) | (uint32_t(tt) << 16) | uint32_t(pos);
    uint32_t h = slot_hash(x, a.log2cap);
    while (atomicCAS(&table[h], kEmpty, e) != kEmpty) h = (h + 1) & mask;
  }
  __syncwarp();

  unsigned char* rec = a.rec + (size_t(bh) * a.T + u) * size_t(a.L.bytes);
  const int me = u - first;  // this token's index in the table
  int fmask = 0;             // bit d: some slot takes a row written d tokens earlier
  for (int e = lane; e < WR; e += 32) {
    int32_t x = e < W ? a.idx_w[(tok0 + u) * W + e] : a.idx_r[(tok0 + u) * R + (e - W)];
    int code = -1;
    if (x < 0 || x >= a.N) {
      code = -2;
      x = 0;
      errs |= SDM_DEV_INDEX_RANGE;
    } else {
      int best_t = -1, best_p = 0;
      for (uint32_t h = slot_hash(x, a.log2cap);; h = (h + 1) & mask) {
        const unsigned long long v = table[h];
        if (v == kEmpty) break;
        if (uint32_t(v >> 32) != uint32_t(x)) continue;
        const int tt = int((v >> 16) & 0xFFFFu), pp = int(v & 0xFFFFu);
        if (e < W && tt == me && pp != e) errs |= SDM_DEV_DUP_WRITE;
        const bool earlier = e < W ? tt < me : tt <= me;
        if (earlier && tt > best_t) {
          best_t = tt;
          best_p = pp;
        }
      }
      if (best_t >= 0) {
        code = (me - best_t) * W + best_p;
        fmask |= 1 << (me - best_t);
      }
    }
    reinterpret_cast<int32_t*>(rec)[e] = x;
    reinterpret_cast<int16_t*>(rec + a.L.off_src)[e] = int16_t(code);
  }
  errs = __reduce_or_sync(0xFFFFFFFFu, errs);
  fmask = __reduce_or_sync(0xFFFFFFFFu, fmask);
  if (errs && lane == 0 && a.dev_err) atomicOr(a.dev_err, errs);

  // Weights, gates and v.
  float* wts = reinterpret_cast<float*>(rec + a.L.off_wts);
  if (reg_softmax) {
    warp_softmax_regs<4>(sw, W, wts);
    warp_softmax_regs<4>(sr, R, wts + W);
  } else {
    warp_softmax(a.sc_w + (tok0 + u) * W, W, wts);
    warp_softmax(a.sc_r + (tok0 + u) * R, R, wts + W);
  }
  if (lane == 0) {
    float* ab = reinterpret_cast<float*>(rec + a.L.off_ab);
    ab[0] = a.alpha[tok0 + u];
    ab[1] = a.beta[tok0 + u];
    reinterpret_cast<int*>(ab)[2] = fmask;
    ab[3] = 0.f;
  }
  float* vr = reinterpret_cast<float*>(rec + a.L.off_v);
  const Tv* vsrc = static_cast<const Tv*>(a.v) + (tok0 + u) * size_t(a.d_v);
  for (int c = lane; c < a.d_v; c += 32) vr[c] = load_v<Tv>(vsrc, c);
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
  pa.BH = BH;
  pa.N = N;
  pa.d_v = d_v;
  pa.W = W;
  pa.R = R;
  pa.pd = pd;
  // The table holds the write sets of pd + 1 tokens and is at most half full.
  int l = 5;
  while ((1LL << l) < 2LL * (pd + 1) * W) ++l;
  pa.log2cap = l;
  pa.L = rec_layout(W, R, d_v);
  pa.rec = static_cast<unsigned char*>(rec);
  pa.dev_err = dev_err;
  int dev = 0, max_smem = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
    return SDM_ECUDA;
  const size_t table = size_t(8) << l;
  pa.warps = int(min(size_t(kPlanMaxWarps), size_t(max_smem) / table));
  if (pa.warps < 1) return SDM_EUNSUPPORTED;
  const size_t smem = size_t(pa.warps) * table;
  const long long blocks = ((long long)BH * T + pa.warps - 1) / pa.warps;
  if (blocks > 0x7FFFFFFFLL) return SDM_EUNSUPPORTED;
  const void* fn = v_dt == SDM_BF16 ? reinterpret_cast<const void*>(&plan_kernel<uint16_t>)
                                    : reinterpret_cast<const void*>(&plan_kernel<float>);
  if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)) != cudaSuccess)
    return SDM_ECUDA;
  void* args[] = {&pa};
  if (cudaLaunchKernel(fn, dim3(unsigned(blocks)), dim3(pa.warps * 32), args, smem, s) != cudaSuccess)
    return SDM_ECUDA;
  return last_launch_status();
}

}  // namespace sdm
