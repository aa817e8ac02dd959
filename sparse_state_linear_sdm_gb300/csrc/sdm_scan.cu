// Recurrent sparse gated-delta scan (Sparse Delta Memory technical summary,
// gist.science/it/paper/2607.07386, "Meccanismo Core" items 3 and 4):
//   M_t[i] = alpha_t M_{t-1}[i] + beta_t k_t^(i) (v_t - alpha_t M_{t-1}[i])  for the W
//   write slots i (k_t: softmax of their scores), all other slots untouched, then
//   o_t = sum_i r_i M_t[i] over the R read slots (r: softmax of their scores).
//
// Two kernels:
//   plan  (time-parallel, one block per (b,h, chunk of tokens)): for every token and
//         every selected slot, finds whether a token at most `pd` steps earlier (or
//         the same token, for a read) wrote that slot, and where in its write set.
//         Also forms both softmaxes and packs slots, weights, alpha, beta and v into
//         one 16-byte-aligned record per token (layout in sdm_internal.cuh).
//   scan  (one block per (b,h, slice of `cols` columns of d_v), sequential in t):
//         the columns of the table are independent given the slots, so each block
//         owns a column slice of one (b,h) table outright.  It gathers the rows of
//         token t+pd from HBM with 16-byte cp.async while it updates token t; rows
//         whose latest writer is still in that window never come from HBM: the
//         writer pushes its updated row into the later token's staging slot
//         (forwarding), which also serves a read of a row written by the same token.
// This is gather/scatter plus axpy: no tensor cores.
#include <cuda_bf16.h>

#include "sdm_internal.cuh"

namespace sdm {
namespace {

constexpr int kPlanThreads = 256;
constexpr int kScanThreads = 256;
constexpr int kScanWarps = kScanThreads / 32;

// Multiplicative hash of a slot into a table of 2^log2cap entries.
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
  int T;
  long long N;
  int d_v, W, R, pd, tc;
  int log2cap;  // hash table of 2^log2cap entries, at least twice the entries inserted
  RecLayout L;
  unsigned char* rec;
  int* dev_err;
};

// Softmax of n scores with one warp, written to w[0..n): one exp per score (the
// unnormalised values are stored first, then scaled in place).
__device__ void warp_softmax(const float* __restrict__ s, int n, float* w) {
  const int lane = threadIdx.x & 31;
  float m = -INFINITY;
  for (int i = lane; i < n; i += 32) m = fmaxf(m, s[i]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, off));
  float z = 0.f;
  for (int i = lane; i < n; i += 32) {
    const float e = expf(s[i] - m);
    w[i] = e;
    z += e;
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) z += __shfl_xor_sync(0xFFFFFFFFu, z, off);
  const float inv = 1.0f / z;
  for (int i = lane; i < n; i += 32) w[i] *= inv;  // each lane rescales what it wrote
}

constexpr unsigned long long kEmpty = ~0ull;

// Shared memory of one planning block: hash table, then the chunk's write slots
// (tokens [t0 - pd, t1)) and read slots (tokens [t0, t1)).
__host__ __device__ inline size_t plan_smem_bytes(int log2cap, int tc, int pd, int W, int R) {
  return (size_t(8) << log2cap) + size_t(tc + pd) * W * 4 + size_t(tc) * R * 4;
}

template <typename Tv>
__global__ void __launch_bounds__(kPlanThreads) plan_kernel(PlanArgs a) {
  // Open-addressing table of the write slots of tokens [tl, t1): one 64-bit word per
  // entry, slot << 32 | (token - tl) << 16 | position in the write set.
  extern __shared__ unsigned long long table[];
  const int tid = threadIdx.x;
  const int bh = blockIdx.y;
  const int t0 = blockIdx.x * a.tc;
  const int t1 = min(a.T, t0 + a.tc);
  const int tl = max(0, t0 - a.pd);
  const int W = a.W, R = a.R, WR = W + R;
  const size_t tok0 = size_t(bh) * a.T;
  const int cap = 1 << a.log2cap, mask = cap - 1;
  int32_t* iw = reinterpret_cast<int32_t*>(table + cap);         // [(t1 - tl) * W]
  int32_t* ir = iw + (a.tc + a.pd) * W;                          // [(t1 - t0) * R]

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
  __syncthreads();
  for (int tt = tl; tt < t1; ++tt) {
    for (int pos = tid; pos < W; pos += kPlanThreads) {
      const int32_t x = iw[(tt - tl) * W + pos];
      if (x < 0 || x >= a.N) continue;
      const unsigned long long e =
          (static_cast<unsigned long long>(uint32_t(x)) << 32) | (uint32_t(tt - tl) << 16) | uint32_t(pos);
      uint32_t h = slot_hash(x, a.log2cap);
      while (atomicCAS(&table[h], kEmpty, e) != kEmpty) h = (h + 1) & mask;
    }
  }
  __syncthreads();

  for (int u = t0; u < t1; ++u) {
    unsigned char* rec = a.rec + (tok0 + u) * size_t(a.L.bytes);
    for (int e = tid; e < WR; e += kPlanThreads) {
      int32_t x = e < W ? iw[(u - tl) * W + e] : ir[(u - t0) * R + (e - W)];
      int code = -1;
      if (x < 0 || x >= a.N) {
        code = -2;
        x = 0;
        if (a.dev_err) atomicOr(a.dev_err, SDM_DEV_INDEX_RANGE);
      } else {
        int best_t = -1, best_p = 0;
        for (uint32_t h = slot_hash(x, a.log2cap);; h = (h + 1) & mask) {
          const unsigned long long v = table[h];
          if (v == kEmpty) break;
          if (uint32_t(v >> 32) != uint32_t(x)) continue;
          const int tt = tl + int((v >> 16) & 0xFFFFu), pp = int(v & 0xFFFFu);
          if (e < W && tt == u && pp != e && a.dev_err) atomicOr(a.dev_err, SDM_DEV_DUP_WRITE);
          const bool earlier = e < W ? tt < u : tt <= u;
          if (earlier && tt >= u - a.pd && tt > best_t) {
            best_t = tt;
            best_p = pp;
          }
        }
        if (best_t >= 0) code = (u - best_t) * W + best_p;
      }
      reinterpret_cast<int32_t*>(rec)[e] = x;
      reinterpret_cast<int16_t*>(rec + a.L.off_src)[e] = int16_t(code);
    }
  }

  // Weights, gates and v for each token of the chunk: one warp per token.
  const int warp = tid >> 5, lane = tid & 31;
  for (int u = t0 + warp; u < t1; u += kPlanThreads / 32) {
    unsigned char* rec = a.rec + (tok0 + u) * size_t(a.L.bytes);
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

// ---------------------------------------------------------------------------------
__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gmem_src) {
  const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(smem_dst));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(d), "l"(gmem_src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;\n" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

struct ScanArgs {
  float* M;
  const unsigned char* rec;
  float* o;
  int T;
  long long N;
  int d_v, W, R;
  RecLayout L;
};

__device__ __forceinline__ float4 f4_add(float4 a, float4 b) {
  return make_float4(a.x + b.x, a.y + b.y, a.z + b.z, a.w + b.w);
}

template <int C, int PD>
__global__ void __launch_bounds__(kScanThreads) scan_kernel(ScanArgs a) {
  constexpr int LPR = C / 4;            // threads per row slice (one float4 each)
  constexpr int RPP = kScanThreads / LPR;  // row slices per pass of the block
  constexpr int MD = 2 * PD;            // records are staged this many tokens ahead
  constexpr int QM = MD + 1;            // record ring slots
  constexpr int QR = PD + 1;            // row ring slots
  extern __shared__ __align__(16) unsigned char smem[];
  const int W = a.W, R = a.R, WR = W + R, T = a.T, d_v = a.d_v;
  const RecLayout L = a.L;
  const int meta_bytes = L.off_v + 4 * C;
  float* rows = reinterpret_cast<float*>(smem);                               // [QR][WR][C]
  unsigned char* meta = smem + size_t(QR) * WR * C * 4;                        // [QM][meta_bytes]
  float* red = reinterpret_cast<float*>(meta + size_t(QM) * meta_bytes);      // [warps][C]

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int slices = d_v / C;
  const int bh = blockIdx.x / slices;
  const int c0 = (blockIdx.x - bh * slices) * C;
  const unsigned char* recs = a.rec + size_t(bh) * T * L.bytes;
  float* Mbh = a.M + size_t(bh) * size_t(a.N) * d_v + c0;
  float* obh = a.o + size_t(bh) * T * d_v + c0;
  const int c4 = tid % LPR;

  auto issue_meta = [&](int u) {
    if (u >= T) return;
    const unsigned char* src = recs + size_t(u) * L.bytes;
    unsigned char* dst = meta + (u % QM) * meta_bytes;
    const int n_main = L.off_v / 16;
    for (int k = tid; k < n_main + LPR; k += kScanThreads) {
      if (k < n_main)
        cp_async16(dst + 16 * k, src + 16 * k);
      else
        cp_async16(dst + L.off_v + 16 * (k - n_main), src + L.off_v + 4 * c0 + 16 * (k - n_main));
    }
  };
  auto issue_rows = [&](int u) {
    if (u >= T) return;
    const unsigned char* mt = meta + (u % QM) * meta_bytes;
    const int32_t* idx = reinterpret_cast<const int32_t*>(mt);
    const int16_t* src = reinterpret_cast<const int16_t*>(mt + L.off_src);
    float* dst = rows + size_t(u % QR) * WR * C;
    for (int k = tid; k < WR * LPR; k += kScanThreads) {
      const int e = k / LPR, q = k % LPR;
      if (src[e] == -1) cp_async16(dst + e * C + 4 * q, Mbh + size_t(idx[e]) * d_v + 4 * q);
    }
  };

  // Prologue: records of tokens [0, PD) first, then the groups the steady state
  // expects from iterations -PD .. -1 (record t+MD, rows t+PD).
  for (int u = 0; u < PD; ++u) issue_meta(u);
  cp_async_commit();
  cp_async_wait<0>();
  __syncthreads();
  for (int j = 0; j < PD; ++j) {
    issue_meta(PD + j);
    cp_async_commit();
    issue_rows(j);
    cp_async_commit();
  }

  for (int t = 0; t < T; ++t) {
    issue_meta(t + MD);
    cp_async_commit();
    // Groups newer than rows(t): 2(PD-1) from iterations t-PD+1 .. t-1 and record(t+MD).
    cp_async_wait<2 * PD - 1>();
    __syncthreads();  // rows(t) and record(t+PD) visible; token t-1 fully retired
    issue_rows(t + PD);
    cp_async_commit();

    const unsigned char* mt = meta + (t % QM) * meta_bytes;
    const int32_t* idx = reinterpret_cast<const int32_t*>(mt);
    const float* wts = reinterpret_cast<const float*>(mt + L.off_wts);
    const int16_t* src = reinterpret_cast<const int16_t*>(mt + L.off_src);
    const float alpha = reinterpret_cast<const float*>(mt + L.off_ab)[0];
    const float beta = reinterpret_cast<const float*>(mt + L.off_ab)[1];
    const float4 vv = reinterpret_cast<const float4*>(mt + L.off_v)[c4];
    float* rs = rows + size_t(t % QR) * WR * C;

    // Forget gate and delta update of the W write rows (in shared memory and in HBM).
    for (int e = tid / LPR; e < W; e += RPP) {
      if (src[e] == -2) continue;
      float4* cell = reinterpret_cast<float4*>(rs + e * C) + c4;
      const float4 m = *cell;
      const float kb = beta * wts[e];
      float4 r;
      float mt_;
      mt_ = alpha * m.x; r.x = fmaf(kb, vv.x - mt_, mt_);
      mt_ = alpha * m.y; r.y = fmaf(kb, vv.y - mt_, mt_);
      mt_ = alpha * m.z; r.z = fmaf(kb, vv.z - mt_, mt_);
      mt_ = alpha * m.w; r.w = fmaf(kb, vv.w - mt_, mt_);
      *cell = r;
      *(reinterpret_cast<float4*>(Mbh + size_t(idx[e]) * d_v) + c4) = r;
    }
    __syncthreads();

    // Forwarding: rows of tokens t .. t+PD whose latest writer is token t.
#pragma unroll
    for (int d = 0; d <= PD; ++d) {
      const int u = t + d;
      if (u >= T) break;
      const unsigned char* mu = meta + (u % QM) * meta_bytes;
      const int16_t* su = reinterpret_cast<const int16_t*>(mu + L.off_src);
      float* ru = rows + size_t(u % QR) * WR * C;
      const int lo = d * W;
      for (int e = (d == 0 ? W : 0) + tid; e < WR; e += kScanThreads) {
        const int code = su[e];
        if (code >= lo && code < lo + W) {
          const float4* from = reinterpret_cast<const float4*>(rs + (code - lo) * C);
          float4* to = reinterpret_cast<float4*>(ru + e * C);
#pragma unroll
          for (int q = 0; q < LPR; ++q) to[q] = from[q];
        }
      }
    }
    __syncthreads();

    // Weighted read of the R read rows (after the write).
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int e = tid / LPR; e < R; e += RPP) {
      if (src[W + e] == -2) continue;
      const float r = wts[W + e];
      const float4 m = reinterpret_cast<const float4*>(rs + (W + e) * C)[c4];
      acc.x = fmaf(r, m.x, acc.x);
      acc.y = fmaf(r, m.y, acc.y);
      acc.z = fmaf(r, m.z, acc.z);
      acc.w = fmaf(r, m.w, acc.w);
    }
#pragma unroll
    for (int off = LPR; off < 32; off <<= 1) {
      acc.x += __shfl_xor_sync(0xFFFFFFFFu, acc.x, off);
      acc.y += __shfl_xor_sync(0xFFFFFFFFu, acc.y, off);
      acc.z += __shfl_xor_sync(0xFFFFFFFFu, acc.z, off);
      acc.w += __shfl_xor_sync(0xFFFFFFFFu, acc.w, off);
    }
    if (lane < LPR) reinterpret_cast<float4*>(red + warp * C)[lane] = acc;
    __syncthreads();
    if (tid < LPR) {
      float4 s = reinterpret_cast<const float4*>(red)[tid];
#pragma unroll
      for (int w = 1; w < kScanWarps; ++w) s = f4_add(s, reinterpret_cast<const float4*>(red + w * C)[tid]);
      *(reinterpret_cast<float4*>(obh + size_t(t) * d_v) + tid) = s;
    }
  }
  cp_async_wait<0>();
}

size_t scan_smem_bytes(int cols, int pd, int W, int R, int d_v) {
  const RecLayout L = rec_layout(W, R, d_v);
  const size_t meta_bytes = size_t(L.off_v) + 4 * size_t(cols);
  return size_t(pd + 1) * (W + R) * cols * 4 + size_t(2 * pd + 1) * meta_bytes +
         size_t(kScanWarps) * cols * 4;
}

using ScanFn = void (*)(ScanArgs);

ScanFn scan_fn(int cols, int pd) {
#define SDM_SCAN_CASE(Cc, Pp) \
  if (cols == Cc && pd == Pp) return &scan_kernel<Cc, Pp>;
  SDM_SCAN_CASE(4, 1) SDM_SCAN_CASE(4, 2) SDM_SCAN_CASE(4, 3)
  SDM_SCAN_CASE(8, 1) SDM_SCAN_CASE(8, 2) SDM_SCAN_CASE(8, 3)
  SDM_SCAN_CASE(16, 1) SDM_SCAN_CASE(16, 2) SDM_SCAN_CASE(16, 3)
  SDM_SCAN_CASE(32, 1) SDM_SCAN_CASE(32, 2) SDM_SCAN_CASE(32, 3)
#undef SDM_SCAN_CASE
  return nullptr;
}

}  // namespace

int choose_scan_shape(int BH, int d_v, int W, int R, int force_cols, int force_pd,
                      ScanShape* out) {
  int dev = 0, max_smem = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return SDM_ECUDA;
  const int col_opts[4] = {32, 16, 8, 4};
  int best_cols = 0, best_pd = 0;
  for (int ci = 0; ci < 4 && !best_cols; ++ci) {
    const int c = col_opts[ci];
    if (force_cols && c != force_cols) continue;
    if (d_v % c) continue;
    // Prefer wide (128-byte) row slices while that still gives ~1.5 blocks per SM.
    if (!force_cols && ci + 1 < 4 && d_v % col_opts[ci + 1] == 0 &&
        (long long)BH * (d_v / c) * 2 < 3LL * sms)
      continue;
    for (int pd = 2; pd >= 1 && !best_cols; --pd) {
      const int p = force_pd ? force_pd : pd;
      if (scan_smem_bytes(c, p, W, R, d_v) <= size_t(max_smem)) {
        best_cols = c;
        best_pd = p;
      }
      if (force_pd) break;
    }
  }
  if (!best_cols) return SDM_EUNSUPPORTED;
  out->cols = best_cols;
  out->pd = best_pd;
  out->blocks = BH * (d_v / best_cols);
  out->smem = int(scan_smem_bytes(best_cols, best_pd, W, R, d_v));
  return SDM_OK;
}

int launch_scan(float* M, const int32_t* idx_w, const float* sc_w, const int32_t* idx_r,
                const float* sc_r, const void* v, int v_dt, const float* alpha, const float* beta,
                int BH, int T, long long N, int d_v, int W, int R, float* o, void* workspace,
                int* dev_err, const ScanShape& shape, cudaEvent_t after_plan, cudaStream_t s) {
  if (T == 0 || BH == 0) return SDM_OK;
  const RecLayout L = rec_layout(W, R, d_v);
  PlanArgs pa;
  pa.idx_w = idx_w;
  pa.sc_w = sc_w;
  pa.idx_r = idx_r;
  pa.sc_r = sc_r;
  pa.v = v;
  pa.alpha = alpha;
  pa.beta = beta;
  pa.T = T;
  pa.N = N;
  pa.d_v = d_v;
  pa.W = W;
  pa.R = R;
  pa.pd = shape.pd;
  // Chunk of tokens per plan block: its write sets (plus pd earlier ones) fill at most
  // half of the hash table, which keeps probe sequences short.
  // Tokens per planning block: at most ~2048 inserted write slots, and shared memory
  // within 96 KB (two blocks per SM); the table has at least twice the inserted entries.
  int tc = 2048 / W - shape.pd;
  tc = tc < 1 ? 1 : (tc > 128 ? 128 : tc);
  auto cap_for = [&](int t) {
    int l = 12;
    while ((1LL << l) < 2LL * (t + shape.pd) * W) ++l;
    return l;
  };
  while (tc > 1 && plan_smem_bytes(cap_for(tc), tc, shape.pd, W, R) > 96 * 1024) --tc;
  pa.tc = tc;
  pa.log2cap = cap_for(tc);
  pa.L = L;
  pa.rec = static_cast<unsigned char*>(workspace);
  pa.dev_err = dev_err;
  const dim3 pgrid((T + tc - 1) / tc, BH);
  const int plan_smem = int(plan_smem_bytes(pa.log2cap, tc, shape.pd, W, R));
  const void* pfn = v_dt == SDM_BF16 ? reinterpret_cast<const void*>(&plan_kernel<uint16_t>)
                                     : reinterpret_cast<const void*>(&plan_kernel<float>);
  if (cudaFuncSetAttribute(pfn, cudaFuncAttributeMaxDynamicSharedMemorySize, plan_smem) !=
      cudaSuccess)
    return SDM_ECUDA;
  if (v_dt == SDM_BF16)
    plan_kernel<uint16_t><<<pgrid, kPlanThreads, plan_smem, s>>>(pa);
  else
    plan_kernel<float><<<pgrid, kPlanThreads, plan_smem, s>>>(pa);
  if (last_launch_status() != SDM_OK) return SDM_ECUDA;
  if (after_plan && cudaEventRecord(after_plan, s) != cudaSuccess) return SDM_ECUDA;

  ScanArgs sa;
  sa.M = M;
  sa.rec = static_cast<const unsigned char*>(workspace);
  sa.o = o;
  sa.T = T;
  sa.N = N;
  sa.d_v = d_v;
  sa.W = W;
  sa.R = R;
  sa.L = L;
  ScanFn fn = scan_fn(shape.cols, shape.pd);
  if (!fn) return SDM_EUNSUPPORTED;
  if (cudaFuncSetAttribute(reinterpret_cast<const void*>(fn),
                           cudaFuncAttributeMaxDynamicSharedMemorySize, shape.smem) != cudaSuccess)
    return SDM_ECUDA;
  fn<<<shape.blocks, kScanThreads, shape.smem, s>>>(sa);
  return last_launch_status();
}

}  // namespace sdm
