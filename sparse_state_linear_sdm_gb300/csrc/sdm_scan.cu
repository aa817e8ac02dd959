// Recurrent sparse gated-delta scan (Sparse Delta Memory technical summary,
// gist.science/it/paper/2607.07386, "Meccanismo Core" items 3 and 4):
//   M_t[i] = alpha_t M_{t-1}[i] + beta_t k_t^(i) (v_t - alpha_t M_{t-1}[i])  for the W
//   write slots i (k_t: softmax of their scores), all other slots untouched, then
//   o_t = sum_i r_i M_t[i] over the R read slots (r: softmax of their scores).
//
// The planning kernel (sdm_plan.cu) first writes one record per token (slots, weights,
// where each row comes from).  The scan kernel here then runs one block per (b, h, slice
// of `cols` columns of d_v), sequential in t: the columns of the table are independent
// given the slots, so each block owns a column slice of one (b, h) table outright.  It
// gathers the rows of token t+pd from HBM with 16-byte cp.async while it updates token t;
// rows whose latest writer is still in that window never come from HBM: the writer
// pushes its updated row into the later token's staging slot (forwarding), which also
// serves a read of a row written by the same token.
// This is gather/scatter plus axpy: no tensor cores.
#include <cuda_bf16.h>

#include "sdm_internal.cuh"

namespace sdm {
namespace {

constexpr int kScanThreads = 256;
constexpr int kScanWarps = kScanThreads / 32;

// ---------------------------------------------------------------------------------
__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gmem_src) {
  const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(smem_dst));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(d), "l"(gmem_src) : "memory");
}
__device__ __forceinline__ void cp_async16_s(uint32_t smem_dst, const void* gmem_src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(smem_dst), "l"(gmem_src) : "memory");
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
  int T;        // tokens of the window
  int T_total;  // tokens per sequence in o
  int t_off;    // first token of the window
  long long N;
  int d_v, W, R;
  RecLayout L;
  float* w_prev;  // optional [BH, T_total, W, d_v]: each write row before its update
  float* r_rows;  // optional [BH, T_total, R, d_v]: each read row as read (after the write)
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
  float* obh = a.o + (size_t(bh) * a.T_total + a.t_off) * d_v + c0;
  float* wsave = a.w_prev ? a.w_prev + (size_t(bh) * a.T_total + a.t_off) * W * d_v + c0 : nullptr;
  float* rsave = a.r_rows ? a.r_rows + (size_t(bh) * a.T_total + a.t_off) * R * d_v + c0 : nullptr;
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
    // Thread tid copies 16-byte chunk c4 of rows tid / LPR + j * RPP: its destination
    // advances by a fixed stride and its source column is fixed.
    uint32_t sdst = static_cast<uint32_t>(
        __cvta_generic_to_shared(rows + size_t(u % QR) * WR * C + (tid / LPR) * C + 4 * c4));
    const float* gcol = Mbh + 4 * c4;
#pragma unroll 4
    for (int e = tid / LPR; e < WR; e += RPP, sdst += RPP * C * 4) {
      if (src[e] == -1) cp_async16_s(sdst, gcol + size_t(idx[e]) * d_v);
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
    // Does a slot of tokens t .. t+PD take a row this token writes?  (bit u - t of record u's
    // forwarding mask; the same answer in every thread.)  Without one, the read rows do not
    // depend on this token's writes and the forwarding step and its barriers are skipped.
    int fwd = 0;
#pragma unroll
    for (int d = 0; d <= PD; ++d)
      if (t + d < T)
        fwd |= (reinterpret_cast<const int*>(meta + ((t + d) % QM) * meta_bytes + L.off_ab)[2] >> d) & 1;

    // Forget gate and delta update of the W write rows (in shared memory and in HBM).
    if (C <= 16 && W <= RPP) {  // narrow slices, at most one row per thread: no batching
      const int e = tid / LPR;
      if (e < W && src[e] != -2) {
        const float4 m = reinterpret_cast<const float4*>(rs + e * C)[c4];
        const float kb = beta * wts[e];
        if (wsave) *(reinterpret_cast<float4*>(wsave + (size_t(t) * W + e) * d_v) + c4) = m;
        float4 r;
        float mt_;
        mt_ = alpha * m.x; r.x = fmaf(kb, vv.x - mt_, mt_);
        mt_ = alpha * m.y; r.y = fmaf(kb, vv.y - mt_, mt_);
        mt_ = alpha * m.z; r.z = fmaf(kb, vv.z - mt_, mt_);
        mt_ = alpha * m.w; r.w = fmaf(kb, vv.w - mt_, mt_);
        reinterpret_cast<float4*>(rs + e * C)[c4] = r;
        *(reinterpret_cast<float4*>(Mbh + size_t(idx[e]) * d_v) + c4) = r;
      }
    } else
    // A thread's rows are distinct, so four of them are read before any is written back:
    // their shared-memory latencies overlap instead of forming one chain.
    for (int e0 = tid / LPR; e0 < W; e0 += 4 * RPP) {
      float4 m[4];
      float kb[4];
      bool ok[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int e = e0 + k * RPP;
        ok[k] = e < W && src[e] != -2;
        if (ok[k]) {
          m[k] = reinterpret_cast<const float4*>(rs + e * C)[c4];
          kb[k] = beta * wts[e];
        }
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        if (!ok[k]) continue;
        const int e = e0 + k * RPP;
        if (wsave) *(reinterpret_cast<float4*>(wsave + (size_t(t) * W + e) * d_v) + c4) = m[k];
        float4 r;
        float mt_;
        mt_ = alpha * m[k].x; r.x = fmaf(kb[k], vv.x - mt_, mt_);
        mt_ = alpha * m[k].y; r.y = fmaf(kb[k], vv.y - mt_, mt_);
        mt_ = alpha * m[k].z; r.z = fmaf(kb[k], vv.z - mt_, mt_);
        mt_ = alpha * m[k].w; r.w = fmaf(kb[k], vv.w - mt_, mt_);
        reinterpret_cast<float4*>(rs + e * C)[c4] = r;
        *(reinterpret_cast<float4*>(Mbh + size_t(idx[e]) * d_v) + c4) = r;
      }
    }

    // Forwarding: rows of tokens t+1 .. t+PD whose latest writer is token t are copied into
    // those tokens' staging slots (their first barrier orders the copies); a read slot of
    // this token that names a row it writes reads the updated row where the write left it.
    // Both need the write phase's rows from every thread: one barrier.
    if (fwd) {
    __syncthreads();
#pragma unroll
    for (int d = 1; d <= PD; ++d) {
      const int u = t + d;
      if (u >= T) break;
      const unsigned char* mu = meta + (u % QM) * meta_bytes;
      const int16_t* su = reinterpret_cast<const int16_t*>(mu + L.off_src);
      float* ru = rows + size_t(u % QR) * WR * C;
      const int lo = d * W;
      for (int e = tid; e < WR; e += kScanThreads) {
        const int code = su[e];
        if (code >= lo && code < lo + W) {
          const float4* from = reinterpret_cast<const float4*>(rs + (code - lo) * C);
          float4* to = reinterpret_cast<float4*>(ru + e * C);
#pragma unroll
          for (int q = 0; q < LPR; ++q) to[q] = from[q];
        }
      }
    }
    }

    // Weighted read of the R read rows (after the write).
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    if (C <= 16 && R <= RPP) {  // narrow slices, at most one row per thread
      const int e = tid / LPR;
      const int code = e < R ? src[W + e] : -2;
      if (code != -2) {
        const float r = wts[W + e];
        const int row = code >= 0 && code < W ? code : W + e;  // this token's write row
        const float4 m = reinterpret_cast<const float4*>(rs + row * C)[c4];
        if (rsave) *(reinterpret_cast<float4*>(rsave + (size_t(t) * R + e) * d_v) + c4) = m;
        acc.x = fmaf(r, m.x, acc.x);
        acc.y = fmaf(r, m.y, acc.y);
        acc.z = fmaf(r, m.z, acc.z);
        acc.w = fmaf(r, m.w, acc.w);
      }
    } else
    for (int e0 = tid / LPR; e0 < R; e0 += 4 * RPP) {  // four rows read, then summed in order
      float4 m[4];
      float r[4];
      bool ok[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int e = e0 + k * RPP;
        const int code = e < R ? src[W + e] : -2;
        ok[k] = code != -2;
        if (ok[k]) {
          r[k] = wts[W + e];
          const int row = code >= 0 && code < W ? code : W + e;  // this token's write row
          m[k] = reinterpret_cast<const float4*>(rs + row * C)[c4];
        }
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        if (!ok[k]) continue;
        if (rsave)
          *(reinterpret_cast<float4*>(rsave + (size_t(t) * R + e0 + k * RPP) * d_v) + c4) = m[k];
        acc.x = fmaf(r[k], m[k].x, acc.x);
        acc.y = fmaf(r[k], m[k].y, acc.y);
        acc.z = fmaf(r[k], m[k].z, acc.z);
        acc.w = fmaf(r[k], m[k].w, acc.w);
      }
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


using ScanFn = void (*)(ScanArgs);

ScanFn scan_fn(int cols, int pd) {
#define SDM_SCAN_CASE(Cc, Pp) \
  if (cols == Cc && pd == Pp) return &scan_kernel<Cc, Pp>;
  SDM_SCAN_CASE(4, 1) SDM_SCAN_CASE(4, 2) SDM_SCAN_CASE(4, 3)
  SDM_SCAN_CASE(8, 1) SDM_SCAN_CASE(8, 2) SDM_SCAN_CASE(8, 3)
  SDM_SCAN_CASE(16, 1) SDM_SCAN_CASE(16, 2) SDM_SCAN_CASE(16, 3)
  SDM_SCAN_CASE(32, 1) SDM_SCAN_CASE(32, 2) SDM_SCAN_CASE(32, 3)
  SDM_SCAN_CASE(64, 1) SDM_SCAN_CASE(64, 2)
#undef SDM_SCAN_CASE
  return nullptr;
}

}  // namespace

size_t scan_smem_bytes(int cols, int pd, int W, int R, int d_v) {
  const RecLayout L = rec_layout(W, R, d_v);
  const size_t meta_bytes = size_t(L.off_v) + 4 * size_t(cols);
  return size_t(pd + 1) * (W + R) * cols * 4 + size_t(2 * pd + 1) * meta_bytes +
         size_t(kScanWarps) * cols * 4;
}

int launch_scan_records(float* M, const void* rec, const TokenWindow& win, long long N, int d_v,
                        int W, int R, float* o, const ScanShape& shape, cudaStream_t s,
                        float* w_prev, float* r_rows) {
  if (win.Tc == 0 || win.BH == 0) return SDM_OK;
  ScanArgs sa;
  sa.M = M;
  sa.rec = static_cast<const unsigned char*>(rec);
  sa.o = o;
  sa.T = win.Tc;
  sa.T_total = win.T_total;
  sa.t_off = win.t0;
  sa.N = N;
  sa.d_v = d_v;
  sa.W = W;
  sa.R = R;
  sa.L = rec_layout(W, R, d_v);
  sa.w_prev = w_prev;
  sa.r_rows = r_rows;
  ScanFn fn = scan_fn(shape.cols, shape.pd);
  if (!fn) return SDM_EUNSUPPORTED;
  if (cudaFuncSetAttribute(reinterpret_cast<const void*>(fn),
                           cudaFuncAttributeMaxDynamicSharedMemorySize, shape.smem) != cudaSuccess)
    return SDM_ECUDA;
  fn<<<win.BH * (d_v / shape.cols), kScanThreads, shape.smem, s>>>(sa);
  return last_launch_status();
}

int launch_scan(float* M, const int32_t* idx_w, const float* sc_w, const int32_t* idx_r,
                const float* sc_r, const void* v, int v_dt, const float* alpha, const float* beta,
                const TokenWindow& win, long long N, int d_v, int W, int R, float* o,
                void* workspace, int* dev_err, const ScanShape& shape, cudaEvent_t after_plan,
                cudaEvent_t wait_before_scan, cudaStream_t s, float* w_prev, float* r_rows) {
  if (win.Tc == 0 || win.BH == 0) return SDM_OK;
  const int st = launch_plan(idx_w, sc_w, idx_r, sc_r, v, v_dt, alpha, beta, win, N, d_v, W, R,
                             shape.pd, workspace, dev_err, s);
  if (st != SDM_OK) return st;
  if (wait_before_scan && cudaStreamWaitEvent(s, wait_before_scan, 0) != cudaSuccess)
    return SDM_ECUDA;
  if (after_plan && cudaEventRecord(after_plan, s) != cudaSuccess) return SDM_ECUDA;
  return launch_scan_records(M, workspace, win, N, d_v, W, R, o, shape, s, w_prev, r_rows);
}

}  // namespace sdm
