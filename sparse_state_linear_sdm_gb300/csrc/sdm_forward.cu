// Pipelined forward pass of one SDM layer (Sparse Delta Memory technical summary,
// gist.science/it/paper/2607.07386, "Meccanismo Core" items 2-4 and "Stato Iniziale
// Appreso"): state from M_0, product-key selection, planning, sparse gated-delta scan.
//
// The selection is compare/select work on the SM cores, the scan and the state
// initialisation are bound by HBM.  Run one after the other they leave either the cores
// or HBM idle, so the sequence is cut into token chunks and four streams overlap them:
//
//   init stream (high priority)    M = M_0 broadcast
//   select stream                  the staircase table (once), then select(0), select(1), ...
//                                  (full-size outputs: never waits)
//   plan stream (high priority)    plan(c) -> record buffer c % 2, after select(c) and
//                                  once scan(c - 2) has consumed that buffer (at low
//                                  priority its small grid waited behind the selection's
//                                  blocks and held up the scans)
//   scan stream (high priority)    scan(c) over record buffer c % 2, after plan(c)
//                                  (the first also after the initialisation)
//
// The selection runs ahead while the state is initialised (the scan cannot start before
// that) and then shares the SMs with the scans.  The scan stream has high priority so that
// its blocks get SM slots ahead of the selection's queue of short blocks.  A chunk boundary is a fresh scan pipeline, exactly as chained calls of
// sdm_scan_forward: the results are bit-identical to the unpipelined path.
//
// The selection blocks read the staircases (the pair-index table of the outer top-K) from a
// table built once per call at the end of the workspace, instead of each block building its
// own in shared memory: with a chunk's few tasks per block that build was a noticeable share
// of the selection.
// The streams and events are created once per device and reused; calls on one device
// are enqueued one at a time (a mutex), and the caller's stream waits for all of the
// call's work before anything enqueued after the call runs.
#include <mutex>

#include "sdm_internal.cuh"

namespace sdm {
namespace {

constexpr int kMaxDevices = 64;
// Automatic chunk size: 512 tokens, or 1024 from 8192 tokens on.  Every chunk's scan launch
// has a fixed cost and the first chunk's selection and planning run before any scan; with 8
// or more chunks of 1024 that head start is amortised and the fewer launches win (B16 H4
// T8192: 25.74-25.79 ms against 26.12-26.15 with 512; 65,536-token calls of the 1M-token
// stream: 946 against 958 ms), with shorter sequences 512 (B4 H8 T2048: 2.03 against 2.06
// ms; B8 H16 T4096: 11.01 against 11.19 ms).
inline int auto_chunk_tokens(int T) { return T >= 8192 ? 1024 : 512; }
constexpr int kMaxChunks = 256;

struct Pipeline {
  bool ready = false;
  cudaStream_t init = nullptr, sel = nullptr, plan = nullptr, scan = nullptr;
  cudaEvent_t start = nullptr, init_done = nullptr, plan_end = nullptr, scan_done = nullptr;
  cudaEvent_t sel_done[2] = {nullptr, nullptr};    // selection of chunk c (c % 2) written
  cudaEvent_t plan_done[2] = {nullptr, nullptr};   // records of buffer i written
  cudaEvent_t buf_free[2] = {nullptr, nullptr};    // records of buffer i consumed
};

std::mutex g_mu;
Pipeline g_pipe[kMaxDevices];

// Streams and events of the current device, created on first use (caller holds g_mu).
int pipeline_of_current_device(Pipeline** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SDM_ECUDA;
  Pipeline& p = g_pipe[dev];
  if (!p.ready) {
    int least = 0, greatest = 0;
    if (cudaDeviceGetStreamPriorityRange(&least, &greatest) != cudaSuccess) return SDM_ECUDA;
    if (cudaStreamCreateWithPriority(&p.init, cudaStreamNonBlocking, greatest) != cudaSuccess ||
        cudaStreamCreateWithPriority(&p.sel, cudaStreamNonBlocking, least) != cudaSuccess ||
        cudaStreamCreateWithPriority(&p.plan, cudaStreamNonBlocking, greatest) != cudaSuccess ||
        cudaStreamCreateWithPriority(&p.scan, cudaStreamNonBlocking, greatest) != cudaSuccess)
      return SDM_ECUDA;
    cudaEvent_t* evs[] = {&p.start,        &p.init_done,    &p.plan_end,    &p.scan_done,
                          &p.sel_done[0],  &p.sel_done[1],  &p.plan_done[0], &p.plan_done[1],
                          &p.buf_free[0],  &p.buf_free[1]};
    for (cudaEvent_t* e : evs)
      if (cudaEventCreateWithFlags(e, cudaEventDisableTiming) != cudaSuccess) return SDM_ECUDA;
    p.ready = true;
  }
  *out = &p;
  return SDM_OK;
}

// Tokens per chunk for a chunk-count request (0 = automatic, about kAutoChunkTokens).
int forward_chunk_tokens(int T, int chunks) {
  if (T <= 0) return 0;
  const int auto_tokens = auto_chunk_tokens(T);
  int n = chunks > 0 ? chunks : (T + auto_tokens - 1) / auto_tokens;
  if (n > kMaxChunks) n = kMaxChunks;
  if (n > T) n = T;
  if (n < 1) n = 1;
  return (T + n - 1) / n;
}

size_t forward_buffer_bytes(int BH, int Tc, int d_v, int W, int R) {
  const size_t b = size_t(BH) * size_t(Tc) * size_t(rec_layout(W, R, d_v).bytes);
  return (b + 255) / 256 * 256;
}

}  // namespace
}  // namespace sdm

using namespace sdm;

extern "C" {

size_t sdm_forward_workspace_size(int B, int H, int T, int d_v, int W, int R, int chunks) {
  if (B < 1 || H < 1 || T < 1 || d_v < 4 || W < 1 || R < 1 || chunks < 0) return 0;
  // two record buffers, then both staircases (sized for min(K, S) = K, the largest)
  return 2 * forward_buffer_bytes(B * H, forward_chunk_tokens(T, chunks), d_v, W, R) +
         (size_t(stair_table_words(W, R, 1 << 20)) * 4 + 255) / 256 * 256;
}

int sdm_forward_chunks(int T, int chunks) {
  if (T < 0 || chunks < 0) return 0;
  const int Tc = forward_chunk_tokens(T, chunks);
  return Tc > 0 ? (T + Tc - 1) / Tc : 0;
}

int sdm_forward_streamed(const void* kp, const void* qp, int in_dt, const void* v, int v_dt,
                         const float* alpha, const float* beta, const float* M0, float* M, int B,
                         int H, int T, int S, int d_v, int W, int R, int32_t* idx_w, float* sc_w,
                         int32_t* idx_r, float* sc_r, float* o, void* workspace,
                         size_t workspace_bytes, int* dev_err, int chunks,
                         void* const* scan_events, void* const* input_ready, void* stream) {
  int st = check_select_args(kp, qp, in_dt, B, H, T, S, W, R, idx_w, sc_w, idx_r, sc_r);
  if (st != SDM_OK) return st;
  const long long N = (long long)S * S;
  st = check_scan_args(M, idx_w, sc_w, idx_r, sc_r, v, v_dt, alpha, beta, B, H, T, N, d_v, W, R,
                       o);
  if (st != SDM_OK) return st;
  if (chunks < 0) return SDM_EINVAL;
  if (M0 && !aligned16(M0)) return SDM_EALIGN;
  if (dev_err && (reinterpret_cast<uintptr_t>(dev_err) & 3u)) return SDM_EALIGN;
  cudaStream_t s = as_stream(stream);
  if (T == 0) return M0 ? launch_init_state(M, M0, B, H, N, d_v, s) : SDM_OK;
  if (!aligned16(workspace)) return SDM_EALIGN;
  if (workspace_bytes < sdm_forward_workspace_size(B, H, T, d_v, W, R, chunks)) return SDM_ENOSPACE;

  const int BH = B * H;
  ScanShape shape;
  st = choose_scan_shape(BH, d_v, W, R, 0, 0, &shape);
  if (st != SDM_OK) return st;
  const int Tc = forward_chunk_tokens(T, chunks);
  const int n = (T + Tc - 1) / Tc;
  const size_t buf = forward_buffer_bytes(BH, Tc, d_v, W, R);
  void* rec[2] = {workspace, static_cast<unsigned char*>(workspace) + buf};
  uint32_t* stairs = reinterpret_cast<uint32_t*>(static_cast<unsigned char*>(workspace) + 2 * buf);

  std::lock_guard<std::mutex> lock(g_mu);
  Pipeline* p = nullptr;
  st = pipeline_of_current_device(&p);
  if (st != SDM_OK) return st;
#define SDM_CK(x) \
  if ((x) != cudaSuccess) return SDM_ECUDA;
  SDM_CK(cudaEventRecord(p->start, s));
  SDM_CK(cudaStreamWaitEvent(p->init, p->start, 0));
  SDM_CK(cudaStreamWaitEvent(p->sel, p->start, 0));
  SDM_CK(cudaStreamWaitEvent(p->plan, p->start, 0));
  st = launch_stair_table(stairs, W, R, S, p->sel);
  if (st != SDM_OK) return st;
  if (M0) {
    st = launch_init_state(M, M0, B, H, N, d_v, p->init);
    if (st != SDM_OK) return st;
  }
  SDM_CK(cudaEventRecord(p->init_done, p->init));
  SDM_CK(cudaStreamWaitEvent(p->scan, p->init_done, 0));
  // Enqueued chunk by chunk, so every wait on a reused event refers to its latest record.
  for (int c = 0; c < n; ++c) {
    const TokenWindow win{BH, (c + 1) * Tc <= T ? Tc : T - c * Tc, T, c * Tc};
    const int b = c & 1;
    // The chunk's k', q', v, alpha, beta may still be arriving (a copy per token window).
    if (input_ready && input_ready[c])
      SDM_CK(cudaStreamWaitEvent(p->sel, static_cast<cudaEvent_t>(input_ready[c]), 0));
    st = in_dt == SDM_BF16
             ? launch_select_bf16(kp, qp, win, S, W, R, idx_w, sc_w, idx_r, sc_r, p->sel, stairs)
             : launch_select_f32(kp, qp, win, S, W, R, idx_w, sc_w, idx_r, sc_r, p->sel, stairs);
    if (st != SDM_OK) return st;
    SDM_CK(cudaEventRecord(p->sel_done[b], p->sel));
    SDM_CK(cudaStreamWaitEvent(p->plan, p->sel_done[b], 0));
    if (c >= 2) SDM_CK(cudaStreamWaitEvent(p->plan, p->buf_free[b], 0));  // scan(c - 2) done
    st = launch_plan(idx_w, sc_w, idx_r, sc_r, v, v_dt, alpha, beta, win, N, d_v, W, R, shape.pd,
                     rec[b], dev_err, p->plan);
    if (st != SDM_OK) return st;
    SDM_CK(cudaEventRecord(p->plan_done[b], p->plan));
    SDM_CK(cudaStreamWaitEvent(p->scan, p->plan_done[b], 0));
    if (scan_events) SDM_CK(cudaEventRecord(static_cast<cudaEvent_t>(scan_events[2 * c]), p->scan));
    st = launch_scan_records(M, rec[b], win, N, d_v, W, R, o, shape, p->scan);
    if (st != SDM_OK) return st;
    if (scan_events)
      SDM_CK(cudaEventRecord(static_cast<cudaEvent_t>(scan_events[2 * c + 1]), p->scan));
    SDM_CK(cudaEventRecord(p->buf_free[b], p->scan));
  }
  // The last plan follows every selection, and the last scan every plan.
  SDM_CK(cudaEventRecord(p->plan_end, p->plan));
  SDM_CK(cudaEventRecord(p->scan_done, p->scan));
  SDM_CK(cudaStreamWaitEvent(s, p->plan_end, 0));
  SDM_CK(cudaStreamWaitEvent(s, p->scan_done, 0));
#undef SDM_CK
  return SDM_OK;
}

int sdm_forward_tuned(const void* kp, const void* qp, int in_dt, const void* v, int v_dt,
                      const float* alpha, const float* beta, const float* M0, float* M, int B,
                      int H, int T, int S, int d_v, int W, int R, int32_t* idx_w, float* sc_w,
                      int32_t* idx_r, float* sc_r, float* o, void* workspace,
                      size_t workspace_bytes, int* dev_err, int chunks, void* const* scan_events,
                      void* stream) {
  return sdm_forward_streamed(kp, qp, in_dt, v, v_dt, alpha, beta, M0, M, B, H, T, S, d_v, W, R,
                              idx_w, sc_w, idx_r, sc_r, o, workspace, workspace_bytes, dev_err,
                              chunks, scan_events, nullptr, stream);
}

int sdm_copy_rows_async(void* dst, size_t dst_pitch, const void* src, size_t src_pitch,
                        size_t row_bytes, size_t rows, void* stream) {
  if (rows == 0 || row_bytes == 0) return SDM_OK;
  if (!dst || !src || dst_pitch < row_bytes || src_pitch < row_bytes) return SDM_EINVAL;
  if (cudaMemcpy2DAsync(dst, dst_pitch, src, src_pitch, row_bytes, rows, cudaMemcpyDefault,
                        as_stream(stream)) != cudaSuccess)
    return SDM_ECUDA;
  return SDM_OK;
}

int sdm_forward(const void* kp, const void* qp, int in_dt, const void* v, int v_dt,
                const float* alpha, const float* beta, const float* M0, float* M, int B, int H,
                int T, int S, int d_v, int W, int R, int32_t* idx_w, float* sc_w, int32_t* idx_r,
                float* sc_r, float* o, void* workspace, size_t workspace_bytes, int* dev_err,
                void* stream) {
  return sdm_forward_tuned(kp, qp, in_dt, v, v_dt, alpha, beta, M0, M, B, H, T, S, d_v, W, R,
                           idx_w, sc_w, idx_r, sc_r, o, workspace, workspace_bytes, dev_err, 0,
                           nullptr, stream);
}

}  // extern "C"
