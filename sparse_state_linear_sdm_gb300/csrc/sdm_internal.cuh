// Internal declarations shared by the SDM CUDA translation units.
#pragma once

#include <cuda_runtime.h>

#include <cmath>
#include <cstddef>
#include <cstdint>

#include "../../include/sdm.h"

namespace sdm {

inline bool aligned16(const void* p) {
  return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
}

inline int last_launch_status() {
  return cudaGetLastError() == cudaSuccess ? SDM_OK : SDM_ECUDA;
}

inline cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }

inline bool bad_dtype(int dt) { return dt != SDM_F32 && dt != SDM_BF16; }

// Argument checks of the selection (sdm_select); pointers only matter when T > 0.
inline int check_select_args(const void* kp, const void* qp, int in_dt, int B, int H, int T,
                             int S, int W, int R, const void* idx_w, const void* sc_w,
                             const void* idx_r, const void* sc_r) {
  if (B < 1 || H < 1 || T < 0 || S < 1 || W < 1 || R < 1 || bad_dtype(in_dt)) return SDM_EINVAL;
  const long long N = (long long)S * S;
  if ((long long)W > N || (long long)R > N) return SDM_EINVAL;
  if (S > SDM_MAX_S || W > SDM_MAX_K || R > SDM_MAX_K) return SDM_EUNSUPPORTED;
  if ((long long)B * H * T > 0x3FFFFFFFFFFFLL) return SDM_EUNSUPPORTED;
  if (T > 0 && (!aligned16(kp) || !aligned16(qp) || !aligned16(idx_w) || !aligned16(sc_w) ||
                !aligned16(idx_r) || !aligned16(sc_r)))
    return SDM_EALIGN;
  return SDM_OK;
}

// Argument checks of the scan (sdm_scan_forward), workspace excluded.
inline int check_scan_args(const float* M, const int32_t* idx_w, const float* sc_w,
                           const int32_t* idx_r, const float* sc_r, const void* v, int v_dt,
                           const float* alpha, const float* beta, int B, int H, int T,
                           long long N, int d_v, int W, int R, const float* o) {
  if (B < 1 || H < 1 || T < 0 || N < 1 || d_v < 4 || d_v % 4 || W < 1 || R < 1) return SDM_EINVAL;
  if (bad_dtype(v_dt) || (long long)W > N || (long long)R > N) return SDM_EINVAL;
  if (W > SDM_MAX_K || R > SDM_MAX_K || d_v > SDM_MAX_DV || N > 0x7FFFFFFFLL)
    return SDM_EUNSUPPORTED;
  if ((long long)B * H > 0x7FFFFFFFLL || (long long)T * (W + R) > 0x7FFFFFFFLL) return SDM_EUNSUPPORTED;
  if (!aligned16(M)) return SDM_EALIGN;
  if (T > 0 && (!aligned16(idx_w) || !aligned16(sc_w) || !aligned16(idx_r) || !aligned16(sc_r) ||
                !aligned16(v) || !aligned16(alpha) || !aligned16(beta) || !aligned16(o)))
    return SDM_EALIGN;
  return SDM_OK;
}

// Per-token record the scan's planning pass writes into the workspace, one per
// (b, h, t).  Every section starts on a 16-byte boundary so the scan can stage it
// with 16-byte asynchronous copies:
//   int32 slot[WRa]     write slots then read slots (W + R entries used)
//   fp32  weight[WRa]   softmax of the write scores, then of the read scores
//   int16 src[WRb]      where the row comes from: -1 = the table in HBM,
//                       -2 = invalid slot (skipped), d*W + p = row p of the write
//                       set of token t-d (0 <= d <= prefetch depth)
//   fp32  alpha, beta; int32 forwarding mask (bit d set: a slot of this token takes the
//         updated row of a write of token t-d); pad
//   fp32  v[d_v]
struct RecLayout {
  int WR, WRa, WRb;
  int off_wts, off_src, off_ab, off_v, bytes;
};

__host__ __device__ inline RecLayout rec_layout(int W, int R, int d_v) {
  RecLayout L;
  L.WR = W + R;
  L.WRa = (L.WR + 3) & ~3;
  L.WRb = (L.WR + 7) & ~7;
  L.off_wts = 4 * L.WRa;
  L.off_src = 8 * L.WRa;
  L.off_ab = L.off_src + 2 * L.WRb;
  L.off_v = L.off_ab + 16;
  L.bytes = L.off_v + 4 * d_v;
  return L;
}

// Bytes of the scan's record workspace, B * H * T records, computed in 64 bits for sizes
// that no check has bounded yet (W, R, d_v taken up to INT_MAX).  False when the product
// does not fit in a size_t.
inline bool scan_workspace_bytes(int B, int H, int T, int d_v, int W, int R, size_t* out) {
  const unsigned long long WR = (unsigned long long)W + (unsigned long long)R;
  const unsigned long long rec = 8 * ((WR + 3) & ~3ull) + 2 * ((WR + 7) & ~7ull) + 16 +
                                 4 * (unsigned long long)d_v;  // rec_layout(W, R, d_v).bytes
  unsigned long long n = 0;
  if (__builtin_mul_overflow((unsigned long long)B, (unsigned long long)H, &n) ||
      __builtin_mul_overflow(n, (unsigned long long)T, &n) || __builtin_mul_overflow(n, rec, &n) ||
      n > (unsigned long long)SIZE_MAX)
    return false;
  *out = size_t(n);
  return true;
}

// Softmax of n scores with one warp (max-subtracted, __expf), written to w[0..n): one exp
// per score (the unnormalised values are stored first, then scaled in place by the lane
// that wrote them).  Shared by the planning kernel (forward weights) and the backward
// kernels, so both see the same weights bit for bit.
__device__ inline void warp_softmax(const float* __restrict__ s, int n, float* w) {
  const int lane = threadIdx.x & 31;
  float m = -INFINITY;
  for (int i = lane; i < n; i += 32) m = fmaxf(m, s[i]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, off));
  float z = 0.f;
  for (int i = lane; i < n; i += 32) {
    const float e = __expf(s[i] - m);
    w[i] = e;
    z += e;
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) z += __shfl_xor_sync(0xFFFFFFFFu, z, off);
  const float inv = 1.0f / z;
  for (int i = lane; i < n; i += 32) w[i] *= inv;
}

// warp_softmax of n <= 32 * E scores held in registers (lane l holds scores l, l + 32, ...;
// entries past n are -inf), with the same operations in the same order, so the weights are
// bit-identical to warp_softmax's.
template <int E>
__device__ inline void warp_softmax_regs(const float (&s)[E], int n, float* w) {
  const int lane = threadIdx.x & 31;
  float m = -INFINITY;
#pragma unroll
  for (int j = 0; j < E; ++j)
    if (lane + 32 * j < n) m = fmaxf(m, s[j]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, off));
  float z = 0.f, e[E];
#pragma unroll
  for (int j = 0; j < E; ++j) {
    e[j] = lane + 32 * j < n ? __expf(s[j] - m) : 0.f;
    if (lane + 32 * j < n) z += e[j];
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) z += __shfl_xor_sync(0xFFFFFFFFu, z, off);
  const float inv = 1.0f / z;
#pragma unroll
  for (int j = 0; j < E; ++j)
    if (lane + 32 * j < n) w[lane + 32 * j] = e[j] * inv;
}

// Tokens [t0, t0 + Tc) of BH sequences stored with T_total tokens each: per-token
// arrays ([BH, T_total, ...]) are read and written in place at token bh * T_total + t;
// planning records are per window, [BH, Tc].
struct TokenWindow {
  int BH;
  int Tc;
  int T_total;
  int t0;
};
inline TokenWindow whole_sequences(int BH, int T) { return TokenWindow{BH, T, T, 0}; }

// Launchers (host side; arguments already validated by the entry points).
int launch_init_state(float* M, const float* M0, int B, int H, long long N, int d_v,
                      cudaStream_t s);
int launch_fill_state(float* M, float value, int B, int H, long long N, int d_v, cudaStream_t s);
int launch_fill_words(int32_t* p, int32_t value, size_t n, cudaStream_t s);
// Both staircases of a (W, R, S) selection into out (stair_table_words 32-bit words).
int stair_table_words(int W, int R, int S);
int launch_stair_table(uint32_t* out, int W, int R, int S, cudaStream_t s);
// Selection kernels of bf16 halves: kSelectAuto = the counting selection where its limits
// hold, else the general one; kSelectGeneral / kSelectCounting force one (the latter
// returns SDM_EUNSUPPORTED outside its limits).
constexpr int kSelectAuto = 0, kSelectGeneral = 1, kSelectCounting = 2;
int launch_select_bf16(const void* kp, const void* qp, const TokenWindow& win, int S, int W,
                       int R, int32_t* idx_w, float* sc_w, int32_t* idx_r, float* sc_r,
                       cudaStream_t s, const uint32_t* stair_g = nullptr, int path = kSelectAuto);
int launch_select_f32(const void* kp, const void* qp, const TokenWindow& win, int S, int W,
                      int R, int32_t* idx_w, float* sc_w, int32_t* idx_r, float* sc_r,
                      cudaStream_t s, const uint32_t* stair_g = nullptr);

// Planning pass of the scan (one record per (b, h, t) of the window into `rec`); `pd` must
// be the prefetch depth of the scan kernel that consumes the records.
int launch_plan(const int32_t* idx_w, const float* sc_w, const int32_t* idx_r, const float* sc_r,
                const void* v, int v_dt, const float* alpha, const float* beta,
                const TokenWindow& win, long long N, int d_v, int W, int R, int pd, void* rec,
                int* dev_err, cudaStream_t s);

struct ScanShape {
  int cols;      // d_v columns per thread block
  int pd;        // prefetch depth (tokens)
  int blocks;
  int smem;      // dynamic shared memory bytes of the scan kernel
};
// Dynamic shared memory of the scan kernel for a column slice and prefetch depth.
size_t scan_smem_bytes(int cols, int pd, int W, int R, int d_v);
// Picks (or checks a forced) scan kernel shape.  Returns SDM_OK or SDM_EUNSUPPORTED.
int choose_scan_shape(int BH, int d_v, int W, int R, int force_cols, int force_pd,
                      ScanShape* out);
// The scan kernel alone, over the window's records (written by launch_plan with the
// same shape.pd); continues from the state in M.
// w_prev / r_rows (optional, [BH, T_total, W or R, d_v]): every write row before its update
// and every read row as read, for the backward pass.
int launch_scan_records(float* M, const void* rec, const TokenWindow& win, long long N, int d_v,
                        int W, int R, float* o, const ScanShape& shape, cudaStream_t s,
                        float* w_prev = nullptr, float* r_rows = nullptr);
// Planning pass, then (after waiting for wait_before_scan, if any, and recording
// after_plan, if any) the scan kernel.
int launch_scan(float* M, const int32_t* idx_w, const float* sc_w, const int32_t* idx_r,
                const float* sc_r, const void* v, int v_dt, const float* alpha, const float* beta,
                const TokenWindow& win, long long N, int d_v, int W, int R, float* o,
                void* workspace, int* dev_err, const ScanShape& shape, cudaEvent_t after_plan,
                cudaEvent_t wait_before_scan, cudaStream_t s, float* w_prev = nullptr,
                float* r_rows = nullptr);

// One decode token (T = 1) of every (b, h) in one kernel: selection, planning and scan.
// SDM_EUNSUPPORTED if its shared memory does not fit (decode_supported: the same check).
int decode_supported(int in_dt, int BH, int S, int d_v, int W, int R);
int launch_decode(const void* kp, const void* qp, int in_dt, const void* v, int v_dt,
                  const float* alpha, const float* beta, float* M, int BH, int S, int d_v, int W,
                  int R, int32_t* idx_w, float* sc_w, int32_t* idx_r, float* sc_r, float* o,
                  int* dev_err, cudaStream_t s, const uint32_t* stairs = nullptr);
// Tests of the projection kernels' timeout path: the producer of cluster rank `cta` (0 for
// the single-CTA kernel) stops issuing copies after `step` K steps, and every wait gives up
// after wait_ns, so that the kernel stops, drains and reports SDM_DEV_TIMEOUT.
struct ProjectStall {
  int cta, step;
  unsigned long long wait_ns;
};
int launch_project(const void* x, const void* w, int B, int T, int D, int H, int S, void* kp,
                   void* qp, int* dev_err, int max_ctas, int pair, cudaStream_t s,
                   const ProjectStall* stall = nullptr);
// Projections fused with the inner top-k of every half, then the outer top-K (two kernels).
size_t project_select_workspace(int B, int T, int H, int S, int W, int R);
int launch_project_select(const void* x, const void* w, int B, int T, int D, int H, int S, int W,
                          int R, int32_t* idx_w, float* sc_w, int32_t* idx_r, float* sc_r,
                          void* workspace, int* dev_err, cudaStream_t s);
// One bounded mbarrier wait of the projection kernel's kind on a single warp (mode 0: never
// completed, 1: completed, 2: stop flag already up); see sdm_test_bounded_wait.
int launch_bounded_wait(int mode, unsigned long long limit_ns, int* dev_err,
                        unsigned long long* elapsed_ns, cudaStream_t s);
int launch_gen_inputs(unsigned long long seed, int B, int H, int T, int b_off, int t_off,
                      long long T_total, int S, int d_v, int in_dt, float alpha_lo,
                      int beta_kind, const float* half_bias, void* kp, void* qp, void* v,
                      float* alpha, float* beta, cudaStream_t s);
int launch_gen_M0(unsigned long long seed, int H, long long N, int d_v, float scale, float* M0,
                  cudaStream_t s);

}  // namespace sdm
