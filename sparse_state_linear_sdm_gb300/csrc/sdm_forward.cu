// Pipelined forward pass of one SDM layer (Sparse Delta Memory technical summary,
// gist.science/it/paper/2607.07386, "Meccanismo Core" items 2-4 and "Stato Iniziale
// Appreso"): state from M_0, product-key selection, planning, sparse gated-delta scan.
//
// The selection is compare/select work on the SM cores, the scan is bound by HBM.  Run one
// after the other they leave either the cores or HBM idle, so the sequence is cut into token
// chunks and four streams overlap them:
//
//   select stream                  select(0), select(1), ... (full-size outputs: never waits)
//   plan stream                    first-writes(c), then plan(c) -> record buffer c % 2,
//                                  after select(c) and once scan(c - 2) has consumed that
//                                  buffer
//   scan stream (high priority)    scan(c) over record buffer c % 2, after plan(c)
//   init stream (high priority)    M_0 into the rows no token writes, after the last
//                                  first-writes pass (beside the remaining scans)
//
// Starting from M_0, the state is not copied before the scan: a row still holds M_0 until
// the first token that writes it, so the planning pass, given each slot's first writing
// token, sends the gathers of rows not yet written to M_0, and the rows never written get
// M_0 at the end.  The scan starts as soon as the first chunk is selected and planned, and
// the copy of M_0 shrinks to the rows no token touches.  Continuing from M (M_0 == NULL)
// skips all of that.  The scan stream has high priority so that its blocks get SM slots
// ahead of the selection's queue of short blocks.  A chunk boundary is a fresh scan
// pipeline, exactly as chained calls of sdm_scan_forward: the results are bit-identical to
// the unpipelined path (state copied from M_0, then one scan).
//
// The streams and events are created once per device and reused; calls on one device
// are enqueued one at a time (a mutex), and the caller's stream waits for all of the
// call's work before anything enqueued after the call runs.
#include <mutex>

#include "sdm_internal.cuh"

namespace sdm {
namespace {

constexpr int kMaxDevices = 64;
constexpr int kAutoChunkTokens = 1024;
constexpr int kMaxChunks = 256;
constexpr int kMaxLead = 6;         // chunks the selection may run ahead of the first scan
constexpr int kSelRing = kMaxLead + 2;
constexpr int kAutoLead = 2;

struct Pipeline {
  bool ready = false;
  cudaStream_t init = nullptr, sel = nullptr, plan = nullptr, scan = nullptr;
  cudaEvent_t start = nullptr, init_done = nullptr, plan_end = nullptr, scan_done = nullptr;
  cudaEvent_t writes_known = nullptr;              // every chunk's first-writes pass done
  cudaEvent_t sel_done[kSelRing] = {};             // selection (and first writes) of chunk c
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
        cudaStreamCreateWithPriority(&p.plan, cudaStreamNonBlocking, least) != cudaSuccess ||
        cudaStreamCreateWithPriority(&p.scan, cudaStreamNonBlocking, greatest) != cudaSuccess)
      return SDM_ECUDA;
    cudaEvent_t* evs[] = {&p.start,        &p.init_done,    &p.plan_end,     &p.scan_done,
                          &p.plan_done[0], &p.plan_done[1], &p.buf_free[0],  &p.buf_free[1],
                          &p.writes_known};
    for (cudaEvent_t* e : evs)
      if (cudaEventCreateWithFlags(e, cudaEventDisableTiming) != cudaSuccess) return SDM_ECUDA;
    for (cudaEvent_t& e : p.sel_done)
      if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) return SDM_ECUDA;
    p.ready = true;
  }
  *out = &p;
  return SDM_OK;
}

// Tokens per chunk for a chunk-count request (0 = automatic, about kAutoChunkTokens).
int forward_chunk_tokens(int T, int chunks) {
  if (T <= 0) return 0;
  int n = chunks > 0 ? chunks : (T + kAutoChunkTokens - 1) / kAutoChunkTokens;
  if (n > kMaxChunks) n = kMaxChunks;
  if (n > T) n = T;
  if (n < 1) n = 1;
  return (T + n - 1) / n;
}

size_t forward_buffer_bytes(int BH, int Tc, int d_v, int W, int R) {
  const size_t b = size_t(BH) * size_t(Tc) * size_t(rec_layout(W, R, d_v).bytes);
  return (b + 255) / 256 * 256;
}

// First-write table: one int32 per (b, h, slot).
size_t first_write_bytes(int BH, long long N) {
  const size_t b = size_t(BH) * size_t(N) * 4;
  return (b + 255) / 256 * 256;
}

}  // namespace
}  // namespace sdm

using namespace sdm;

extern "C" {

size_t sdm_forward_workspace_size(int B, int H, int T, int S, int d_v, int W, int R, int chunks) {
  if (B < 1 || H < 1 || T < 1 || S < 1 || d_v < 4 || W < 1 || R < 1 || chunks < 0) return 0;
  return 2 * forward_buffer_bytes(B * H, forward_chunk_tokens(T, chunks), d_v, W, R) +
         first_write_bytes(B * H, (long long)S * S);
}

int sdm_forward_chunks(int T, int chunks) {
  if (T < 0 || chunks < 0) return 0;
  const int Tc = forward_chunk_tokens(T, chunks);
  return Tc > 0 ? (T + Tc - 1) / Tc : 0;
}

int sdm_forward_tuned(const void* kp, const void* qp, int in_dt, const void* v, int v_dt,
                      const float* alpha, const float* beta, const float* M0, float* M, int B,
                      int H, int T, int S, int d_v, int W, int R, int32_t* idx_w, float* sc_w,
                      int32_t* idx_r, float* sc_r, float* o, void* workspace,
                      size_t workspace_bytes, int* dev_err, int chunks, int lead,
                      void* const* scan_events, void* stream) {
  int st = check_select_args(kp, qp, in_dt, B, H, T, S, W, R, idx_w, sc_w, idx_r, sc_r);
  if (st != SDM_OK) return st;
  const long long N = (long long)S * S;
  st = check_scan_args(M, idx_w, sc_w, idx_r, sc_r, v, v_dt, alpha, beta, B, H, T, N, d_v, W, R,
                       o);
  if (st != SDM_OK) return st;
  if (chunks < 0 || lead < -1 || lead > kMaxLead) return SDM_EINVAL;
  if (M0 && !aligned16(M0)) return SDM_EALIGN;
  if (dev_err && (reinterpret_cast<uintptr_t>(dev_err) & 3u)) return SDM_EALIGN;
  cudaStream_t s = as_stream(stream);
  if (T == 0) return M0 ? launch_init_state(M, M0, B, H, N, d_v, s) : SDM_OK;
  if (!aligned16(workspace)) return SDM_EALIGN;
  if (workspace_bytes < sdm_forward_workspace_size(B, H, T, S, d_v, W, R, chunks))
    return SDM_ENOSPACE;

  const int BH = B * H;
  ScanShape shape;
  st = choose_scan_shape(BH, d_v, W, R, 0, 0, &shape);
  if (st != SDM_OK) return st;
  const int Tc = forward_chunk_tokens(T, chunks);
  const int n = (T + Tc - 1) / Tc;
  const size_t buf = forward_buffer_bytes(BH, Tc, d_v, W, R);
  void* rec[2] = {workspace, static_cast<unsigned char*>(workspace) + buf};
  int32_t* first =
      M0 ? reinterpret_cast<int32_t*>(static_cast<unsigned char*>(workspace) + 2 * buf) : nullptr;

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
  SDM_CK(cudaStreamWaitEvent(p->scan, p->start, 0));
  if (first)
    SDM_CK(cudaMemsetAsync(first, 0x7F, first_write_bytes(BH, N), p->sel));  // kNeverWritten
  // The selection runs `ld` chunks ahead of the first scan: it is issue-bound like the scan
  // and gets few SM slots once the scans run, so it is given a head start.
  const int ld = lead < 0 ? kAutoLead : lead;
  auto select_chunk = [&](int c) -> int {
    const TokenWindow win{BH, (c + 1) * Tc <= T ? Tc : T - c * Tc, T, c * Tc};
    int r = in_dt == SDM_BF16
                ? launch_select_bf16(kp, qp, win, S, W, R, idx_w, sc_w, idx_r, sc_r, p->sel)
                : launch_select_f32(kp, qp, win, S, W, R, idx_w, sc_w, idx_r, sc_r, p->sel);
    if (r != SDM_OK) return r;
    if (first) {
      r = launch_first_writes(idx_w, win, N, W, first, p->sel);
      if (r != SDM_OK) return r;
      if (c == n - 1 && cudaEventRecord(p->writes_known, p->sel) != cudaSuccess) return SDM_ECUDA;
    }
    return cudaEventRecord(p->sel_done[c % kSelRing], p->sel) == cudaSuccess ? SDM_OK : SDM_ECUDA;
  };
  // Enqueued chunk by chunk, so every wait on a reused event refers to its latest record.
  for (int c = 0; c < n && c < ld; ++c)
    if ((st = select_chunk(c)) != SDM_OK) return st;
  for (int c = 0; c < n; ++c) {
    const TokenWindow win{BH, (c + 1) * Tc <= T ? Tc : T - c * Tc, T, c * Tc};
    const int b = c & 1;
    if (c + ld < n && (st = select_chunk(c + ld)) != SDM_OK) return st;
    if (c == 0) SDM_CK(cudaStreamWaitEvent(p->scan, p->sel_done[(n - 1 < ld ? n - 1 : ld) % kSelRing], 0));
    SDM_CK(cudaStreamWaitEvent(p->plan, p->sel_done[c % kSelRing], 0));
    if (c >= 2) SDM_CK(cudaStreamWaitEvent(p->plan, p->buf_free[b], 0));  // scan(c - 2) done
    st = launch_plan(idx_w, sc_w, idx_r, sc_r, v, v_dt, alpha, beta, win, N, d_v, W, R, shape.pd,
                     rec[b], dev_err, p->plan, first);
    if (st != SDM_OK) return st;
    SDM_CK(cudaEventRecord(p->plan_done[b], p->plan));
    SDM_CK(cudaStreamWaitEvent(p->scan, p->plan_done[b], 0));
    if (scan_events) SDM_CK(cudaEventRecord(static_cast<cudaEvent_t>(scan_events[2 * c]), p->scan));
    st = launch_scan_records(M, rec[b], win, N, d_v, W, R, o, shape, p->scan, nullptr, nullptr,
                             M0, H);
    if (st != SDM_OK) return st;
    if (scan_events)
      SDM_CK(cudaEventRecord(static_cast<cudaEvent_t>(scan_events[2 * c + 1]), p->scan));
    SDM_CK(cudaEventRecord(p->buf_free[b], p->scan));
  }
  if (first) {  // rows no token writes: M_0, beside the scans still running (disjoint rows)
    SDM_CK(cudaStreamWaitEvent(p->init, p->writes_known, 0));
    st = launch_fill_unwritten(M, M0, first, B, H, N, d_v, p->init);
    if (st != SDM_OK) return st;
  }
  SDM_CK(cudaEventRecord(p->init_done, p->init));
  SDM_CK(cudaStreamWaitEvent(s, p->init_done, 0));
  // The last plan follows every selection, and the last scan every plan.
  SDM_CK(cudaEventRecord(p->plan_end, p->plan));
  SDM_CK(cudaEventRecord(p->scan_done, p->scan));
  SDM_CK(cudaStreamWaitEvent(s, p->plan_end, 0));
  SDM_CK(cudaStreamWaitEvent(s, p->scan_done, 0));
#undef SDM_CK
  return SDM_OK;
}

int sdm_forward(const void* kp, const void* qp, int in_dt, const void* v, int v_dt,
                const float* alpha, const float* beta, const float* M0, float* M, int B, int H,
                int T, int S, int d_v, int W, int R, int32_t* idx_w, float* sc_w, int32_t* idx_r,
                float* sc_r, float* o, void* workspace, size_t workspace_bytes, int* dev_err,
                void* stream) {
  return sdm_forward_tuned(kp, qp, in_dt, v, v_dt, alpha, beta, M0, M, B, H, T, S, d_v, W, R,
                           idx_w, sc_w, idx_r, sc_r, o, workspace, workspace_bytes, dev_err, 0,
                           -1, nullptr, stream);
}

}  // extern "C"
