// C ABI entry points of the SDM forward hot path: host-side argument checks, then
// the launchers.  Nothing here allocates device memory or keeps pointers.
#include "sdm_internal.cuh"

using namespace sdm;


extern "C" {

const char* sdm_status_str(int status) {
  switch (status) {
    case SDM_OK: return "ok";
    case SDM_EINVAL: return "invalid argument (size or dtype out of range)";
    case SDM_EALIGN: return "pointer is NULL or not 16-byte aligned";
    case SDM_ECUDA: return "CUDA launch or query failed";
    case SDM_ETIMEOUT: return "bounded device wait ran out";
    case SDM_EBOUNDS: return "device-detected bounds error";
    case SDM_EUNSUPPORTED: return "sizes beyond the library's limits";
    case SDM_ENOSPACE: return "workspace smaller than required";
    case SDM_ESCRATCH: return "problem too large for the fixed no-allocation scratch";
    default: return "unknown status";
  }
}

int sdm_init_state_from_M0(float* M, const float* M0, int B, int H, long long N, int d_v,
                           void* stream) {
  if (B < 1 || H < 1 || N < 1 || d_v < 4 || d_v % 4) return SDM_EINVAL;
  if (!aligned16(M) || !aligned16(M0)) return SDM_EALIGN;
  return launch_init_state(M, M0, B, H, N, d_v, as_stream(stream));
}

int sdm_fill_state(float* M, float value, int B, int H, long long N, int d_v, void* stream) {
  if (B < 1 || H < 1 || N < 1 || d_v < 4 || d_v % 4) return SDM_EINVAL;
  if (!aligned16(M)) return SDM_EALIGN;
  return launch_fill_state(M, value, B, H, N, d_v, as_stream(stream));
}

int sdm_select_tuned(const void* kp, const void* qp, int in_dt, int B, int H, int T, int S, int W,
                     int R, int32_t* idx_w, float* sc_w, int32_t* idx_r, float* sc_r, int path,
                     void* stream) {
  const int st = check_select_args(kp, qp, in_dt, B, H, T, S, W, R, idx_w, sc_w, idx_r, sc_r);
  if (st != SDM_OK) return st;
  if (path < kSelectAuto || path > kSelectCounting) return SDM_EINVAL;
  if (in_dt != SDM_BF16 && path == kSelectCounting) return SDM_EUNSUPPORTED;
  if (T == 0) return SDM_OK;
  return in_dt == SDM_BF16
             ? launch_select_bf16(kp, qp, whole_sequences(B * H, T), S, W, R, idx_w, sc_w, idx_r,
                                  sc_r, as_stream(stream), nullptr, path)
             : launch_select_f32(kp, qp, whole_sequences(B * H, T), S, W, R, idx_w, sc_w, idx_r,
                                 sc_r, as_stream(stream));
}

int sdm_select(const void* kp, const void* qp, int in_dt, int B, int H, int T, int S, int W, int R,
               int32_t* idx_w, float* sc_w, int32_t* idx_r, float* sc_r, void* stream) {
  return sdm_select_tuned(kp, qp, in_dt, B, H, T, S, W, R, idx_w, sc_w, idx_r, sc_r, kSelectAuto,
                          stream);
}

int sdm_decode_step(const void* kp, const void* qp, int in_dt, const void* v, int v_dt,
                    const float* alpha, const float* beta, float* M, int B, int H, int S, int d_v,
                    int W, int R, int32_t* idx_w, float* sc_w, int32_t* idx_r, float* sc_r,
                    float* o, int* dev_err, void* stream) {
  return sdm_decode_step_tabled(kp, qp, in_dt, v, v_dt, alpha, beta, M, B, H, S, d_v, W, R, idx_w,
                                sc_w, idx_r, sc_r, o, dev_err, nullptr, stream);
}

int sdm_decode_table_words(int W, int R, int S) {
  if (W < 1 || R < 1 || S < 1 || S > SDM_MAX_S || W > SDM_MAX_K || R > SDM_MAX_K) return -1;
  return stair_table_words(W, R, S);
}

int sdm_decode_table(uint32_t* table, int W, int R, int S, void* stream) {
  if (sdm_decode_table_words(W, R, S) < 0) return SDM_EINVAL;
  if (!table) return SDM_EINVAL;
  if (reinterpret_cast<uintptr_t>(table) & 3u) return SDM_EALIGN;
  return launch_stair_table(table, W, R, S, as_stream(stream));
}

int sdm_decode_step_tabled(const void* kp, const void* qp, int in_dt, const void* v, int v_dt,
                           const float* alpha, const float* beta, float* M, int B, int H, int S,
                           int d_v, int W, int R, int32_t* idx_w, float* sc_w, int32_t* idx_r,
                           float* sc_r, float* o, int* dev_err, const uint32_t* table,
                           void* stream) {
  if (table && (reinterpret_cast<uintptr_t>(table) & 3u)) return SDM_EALIGN;
  int st = check_select_args(kp, qp, in_dt, B, H, 1, S, W, R, idx_w, sc_w, idx_r, sc_r);
  if (st != SDM_OK) return st;
  const long long N = (long long)S * S;
  st = check_scan_args(M, idx_w, sc_w, idx_r, sc_r, v, v_dt, alpha, beta, B, H, 1, N, d_v, W, R,
                       o);
  if (st != SDM_OK) return st;
  if (dev_err && (reinterpret_cast<uintptr_t>(dev_err) & 3u)) return SDM_EALIGN;
  return launch_decode(kp, qp, in_dt, v, v_dt, alpha, beta, M, B * H, S, d_v, W, R, idx_w, sc_w,
                       idx_r, sc_r, o, dev_err, as_stream(stream), table);
}

int sdm_decode_step_supported(int in_dt, int B, int H, int S, int d_v, int W, int R) {
  if (bad_dtype(in_dt) || B < 1 || H < 1 || S < 1 || S > SDM_MAX_S || d_v < 4 || d_v % 4 ||
      W < 1 || R < 1 || W > SDM_MAX_K || R > SDM_MAX_K || 1LL * W > 1LL * S * S ||
      1LL * R > 1LL * S * S)
    return SDM_EINVAL;
  return decode_supported(in_dt, B * H, S, d_v, W, R);
}

size_t sdm_project_select_workspace_size(int B, int T, int H, int S, int W, int R) {
  if (B < 1 || T < 1 || H < 1 || S < 1 || W < 1 || R < 1) return 0;
  return project_select_workspace(B, T, H, S, W, R);
}

int sdm_project_select(const void* x, const void* w, int B, int T, int D, int H, int S, int W,
                       int R, int32_t* idx_w, float* sc_w, int32_t* idx_r, float* sc_r,
                       void* workspace, size_t workspace_bytes, int* dev_err, void* stream) {
  if (B < 1 || T < 1 || H < 1 || S < 1 || D < 8 || D % 8 || W < 1 || R < 1) return SDM_EINVAL;
  if (1LL * W > 1LL * S * S || 1LL * R > 1LL * S * S) return SDM_EINVAL;
  if (S % 128 || S > 1024 || W > 128 || R > 128) return SDM_EUNSUPPORTED;
  if (1LL * B * T >= (1LL << 31) || 4LL * H * S >= (1LL << 31)) return SDM_EUNSUPPORTED;
  if (!aligned16(x) || !aligned16(w) || !aligned16(idx_w) || !aligned16(sc_w) || !aligned16(idx_r) ||
      !aligned16(sc_r) || !aligned16(workspace))
    return SDM_EALIGN;
  if (dev_err && (reinterpret_cast<uintptr_t>(dev_err) & 3u)) return SDM_EALIGN;
  if (workspace_bytes < project_select_workspace(B, T, H, S, W, R)) return SDM_ENOSPACE;
  return launch_project_select(x, w, B, T, D, H, S, W, R, idx_w, sc_w, idx_r, sc_r, workspace,
                               dev_err, as_stream(stream));
}

int sdm_project_kq_tuned(const void* x, const void* w, int B, int T, int D, int H, int S,
                         void* kp, void* qp, int* dev_err, int max_ctas, int pair, void* stream) {
  if (B < 1 || T < 1 || H < 1 || S < 1 || D < 8 || D % 8 || max_ctas < 0 ||
      (pair != -1 && pair != 0 && pair != 2))
    return SDM_EINVAL;
  if (S > SDM_MAX_S) return SDM_EUNSUPPORTED;
  if (1LL * B * T >= (1LL << 31) || 4LL * H * S >= (1LL << 31)) return SDM_EUNSUPPORTED;
  if (!aligned16(x) || !aligned16(w) || !aligned16(kp) || !aligned16(qp)) return SDM_EALIGN;
  if (dev_err && (reinterpret_cast<uintptr_t>(dev_err) & 3u)) return SDM_EALIGN;
  return launch_project(x, w, B, T, D, H, S, kp, qp, dev_err, max_ctas, pair, as_stream(stream));
}

int sdm_project_kq(const void* x, const void* w, int B, int T, int D, int H, int S, void* kp,
                   void* qp, int* dev_err, void* stream) {
  return sdm_project_kq_tuned(x, w, B, T, D, H, S, kp, qp, dev_err, 0, -1, stream);
}

int sdm_test_project_stall(const void* x, const void* w, int B, int T, int D, int H, int S,
                           void* kp, void* qp, int pair, int stall_cta, int stall_step,
                           unsigned long long wait_ns, int* dev_err, void* stream) {
  if (B < 1 || T < 1 || H < 1 || S < 1 || D < 8 || D % 8 || (pair != 0 && pair != 2) ||
      stall_cta < 0 || stall_cta > (pair == 2 ? 1 : 0) || stall_step < 0 || wait_ns < 100000ull ||
      wait_ns > 1000000000ull || !dev_err)
    return SDM_EINVAL;
  if (S > SDM_MAX_S) return SDM_EUNSUPPORTED;
  if (1LL * B * T >= (1LL << 31) || 4LL * H * S >= (1LL << 31)) return SDM_EUNSUPPORTED;
  if (pair == 2 && 1LL * B * T <= 128) return SDM_EUNSUPPORTED;  // one row tile: no pair
  if (!aligned16(x) || !aligned16(w) || !aligned16(kp) || !aligned16(qp)) return SDM_EALIGN;
  if (reinterpret_cast<uintptr_t>(dev_err) & 3u) return SDM_EALIGN;
  const ProjectStall stall{stall_cta, stall_step, wait_ns};
  return launch_project(x, w, B, T, D, H, S, kp, qp, dev_err, 0, pair, as_stream(stream), &stall);
}

int sdm_test_bounded_wait(int mode, unsigned long long limit_ns, int* dev_err,
                          unsigned long long* elapsed_ns, void* stream) {
  if (mode < 0 || mode > 2 || limit_ns > 1000000000ull || !dev_err) return SDM_EINVAL;
  if (reinterpret_cast<uintptr_t>(dev_err) & 3u) return SDM_EALIGN;
  if (elapsed_ns && (reinterpret_cast<uintptr_t>(elapsed_ns) & 7u)) return SDM_EALIGN;
  return launch_bounded_wait(mode, limit_ns, dev_err, elapsed_ns, as_stream(stream));
}

size_t sdm_scan_workspace_size(int B, int H, int T, int d_v, int W, int R) {
  if (B < 1 || H < 1 || T < 1 || d_v < 4 || W < 1 || R < 1) return 0;
  size_t bytes = 0;
  return scan_workspace_bytes(B, H, T, d_v, W, R, &bytes) ? bytes : SIZE_MAX;
}

int sdm_scan_forward_tuned(float* M, const int32_t* idx_w, const float* sc_w,
                           const int32_t* idx_r, const float* sc_r, const void* v, int v_dt,
                           const float* alpha, const float* beta, int B, int H, int T,
                           long long N, int d_v, int W, int R, float* o, void* workspace,
                           size_t workspace_bytes, int* dev_err, int cols_per_cta,
                           int prefetch_depth, void* event_after_plan, void* wait_before_scan,
                           void* stream) {
  int st = check_scan_args(M, idx_w, sc_w, idx_r, sc_r, v, v_dt, alpha, beta, B, H, T, N, d_v, W,
                           R, o);
  if (st != SDM_OK) return st;
  if (cols_per_cta < 0 || prefetch_depth < 0 || prefetch_depth > 3) return SDM_EINVAL;
  if (T == 0) return SDM_OK;
  if (!aligned16(workspace)) return SDM_EALIGN;
  if (workspace_bytes < sdm_scan_workspace_size(B, H, T, d_v, W, R)) return SDM_ENOSPACE;
  if (dev_err && (reinterpret_cast<uintptr_t>(dev_err) & 3u)) return SDM_EALIGN;
  ScanShape shape;
  st = choose_scan_shape(B * H, d_v, W, R, cols_per_cta, prefetch_depth, &shape);
  if (st != SDM_OK) return st;
  return launch_scan(M, idx_w, sc_w, idx_r, sc_r, v, v_dt, alpha, beta, whole_sequences(B * H, T),
                     N, d_v, W, R, o, workspace, dev_err, shape,
                     reinterpret_cast<cudaEvent_t>(event_after_plan),
                     reinterpret_cast<cudaEvent_t>(wait_before_scan), as_stream(stream));
}

int sdm_scan_forward(float* M, const int32_t* idx_w, const float* sc_w, const int32_t* idx_r,
                     const float* sc_r, const void* v, int v_dt, const float* alpha,
                     const float* beta, int B, int H, int T, long long N, int d_v, int W, int R,
                     float* o, void* workspace, size_t workspace_bytes, int* dev_err,
                     void* stream) {
  return sdm_scan_forward_tuned(M, idx_w, sc_w, idx_r, sc_r, v, v_dt, alpha, beta, B, H, T, N, d_v,
                                W, R, o, workspace, workspace_bytes, dev_err, 0, 0, nullptr, nullptr,
                                stream);
}

int sdm_scan_launch_info(int B, int H, int d_v, int W, int R, int* cols_per_cta,
                         int* prefetch_depth, int* blocks, int* smem_bytes) {
  if (B < 1 || H < 1 || d_v < 4 || d_v % 4 || W < 1 || R < 1) return SDM_EINVAL;
  if (W > SDM_MAX_K || R > SDM_MAX_K) return SDM_EUNSUPPORTED;
  ScanShape shape;
  const int st = choose_scan_shape(B * H, d_v, W, R, 0, 0, &shape);
  if (st != SDM_OK) return st;
  if (cols_per_cta) *cols_per_cta = shape.cols;
  if (prefetch_depth) *prefetch_depth = shape.pd;
  if (blocks) *blocks = shape.blocks;
  if (smem_bytes) *smem_bytes = shape.smem;
  return SDM_OK;
}

int sdm_gen_inputs(unsigned long long seed, int B, int H, int T, int b_off, int t_off,
                   long long T_total, int S, int d_v, int in_dt, float alpha_lo, int beta_kind,
                   const float* half_bias, void* kp, void* qp, void* v, float* alpha,
                   float* beta, void* stream) {
  if (B < 0 || H < 1 || T < 0 || b_off < 0 || t_off < 0 || S < 1 || d_v < 1 || bad_dtype(in_dt))
    return SDM_EINVAL;
  if ((long long)t_off + T > T_total || (beta_kind != 0 && beta_kind != 1)) return SDM_EINVAL;
  if (!(alpha_lo >= 0.0f && alpha_lo <= 1.0f)) return SDM_EINVAL;
  const void* ptrs[6] = {kp, qp, v, alpha, beta, half_bias};
  for (const void* p : ptrs)
    if (p && (reinterpret_cast<uintptr_t>(p) & 3u)) return SDM_EALIGN;
  return launch_gen_inputs(seed, B, H, T, b_off, t_off, T_total, S, d_v, in_dt, alpha_lo,
                           beta_kind, half_bias, kp, qp, v, alpha, beta, as_stream(stream));
}

int sdm_gen_M0(unsigned long long seed, int H, long long N, int d_v, float scale, float* M0,
               void* stream) {
  if (H < 1 || N < 1 || d_v < 1) return SDM_EINVAL;
  if (!aligned16(M0)) return SDM_EALIGN;
  return launch_gen_M0(seed, H, N, d_v, scale, M0, as_stream(stream));
}

}  // extern "C"
