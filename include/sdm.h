/* sdm.h - C ABI of the GB300 (sm_103a) Sparse Delta Memory forward hot path.
 *
 * The layer (Sparse Delta Memory (SDM) technical summary,
 * gist.science/it/paper/2607.07386, "Meccanismo Core" items 1-4):
 *   each (sequence b, head h) owns a memory table M in R^{N x d_v}, started from a
 *   learned M_0 ("Stato Iniziale Appreso").  At every token t the projected key k'
 *   and query q' are split in two halves of S = sqrt(N) sub-scores each; slot
 *   i*S + j scores half0[i] + half1[j].  The top-W slots of k' are written with
 *     M_t[i] = alpha_t M_{t-1}[i] + beta_t k_t^(i) (v_t - alpha_t M_{t-1}[i])
 *   (k_t^(i): softmax over the W selected write scores), every other slot is left
 *   untouched, and the output is o_t = sum_i r_i M_t[i] over the top-R slots of q'
 *   (r: softmax over the R selected read scores), read after the write.
 *
 * Conventions for every entry point:
 *   - All tensor pointers are DEVICE pointers owned by the caller; the library
 *     keeps no pointer after the call returns and allocates nothing.  Tensors are
 *     dense row-major ("C order") with the shapes given below and must be 16-byte
 *     aligned (SDM_EALIGN otherwise).
 *   - `stream` is a cudaStream_t passed as a plain pointer (NULL = legacy default
 *     stream).  Work is enqueued asynchronously on it; the call returns before the
 *     GPU finishes.
 *   - Arguments are checked on the host before anything is launched.  A failed
 *     check returns SDM_EINVAL / SDM_EALIGN / SDM_EUNSUPPORTED and launches
 *     nothing.  A failed launch returns SDM_ECUDA (cudaGetLastError is consumed).
 *   - Conditions only the GPU can see (a slot index outside [0, N), a repeated slot
 *     in one token's write set) are OR-ed into `*dev_err` (SDM_DEV_* bits, device
 *     memory, may be NULL) and never trap; the offending rows are skipped, so no
 *     access leaves the caller's buffers, and the results are then unspecified.
 *   - Floating-point inputs are expected finite; NaN sub-scores give an
 *     unspecified selection.
 */
#ifndef SDM_H_
#define SDM_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  SDM_OK = 0,
  SDM_EINVAL = -1,       /* a size or dtype argument is out of range */
  SDM_EALIGN = -2,       /* a pointer is NULL or not 16-byte aligned */
  SDM_ECUDA = -3,        /* a CUDA launch or query failed */
  SDM_ETIMEOUT = -4,     /* reserved: a bounded device wait ran out */
  SDM_EBOUNDS = -5,      /* reserved: device-detected bounds error */
  SDM_EUNSUPPORTED = -6, /* sizes valid for the method but beyond the library's limits */
  SDM_ENOSPACE = -7,     /* the workspace passed is smaller than required */
  SDM_ESCRATCH = -8      /* too large for sdm_scan_forward_noalloc's fixed scratch */
} sdm_status;

typedef enum { SDM_F32 = 0, SDM_BF16 = 1 } sdm_dtype;

/* bits OR-ed into *dev_err by the device */
#define SDM_DEV_INDEX_RANGE 1 /* a slot index was < 0 or >= N */
#define SDM_DEV_DUP_WRITE 2   /* a slot appeared twice in one token's write set */
#define SDM_DEV_TIMEOUT 4     /* a bounded wait inside a kernel ran out; outputs unspecified */

/* Limits of the library (checked on the host, SDM_EUNSUPPORTED beyond them). */
#define SDM_MAX_S 4096   /* sqrt(N) */
#define SDM_MAX_K 1024   /* W and R */
#define SDM_MAX_DV 65536 /* d_v of the scan entry points */

/* Human-readable name of a status code (static string). */
const char* sdm_status_str(int status);

/* sdm_init_state_from_M0 - start every sequence from the learned initial state
 * ("Stato Iniziale Appreso": M_0 is a learnable parameter copied into the state).
 *   M  [B, H, N, d_v] fp32, written: M[b, h] = M0[h] for every b.
 *   M0 [H, N, d_v]    fp32, read only.
 * Requires B, H >= 1, N >= 1, d_v >= 4, d_v % 4 == 0. */
int sdm_init_state_from_M0(float* M, const float* M0, int B, int H, long long N, int d_v,
                           void* stream);

/* sdm_fill_state - every entry of a state-shaped table set to `value` (not the method itself:
 * the backward pass's adjoint table starts at zero when the final state carries no gradient,
 * see sdm_scan_backward).  M [B, H, N, d_v] fp32, written with streaming stores.
 * Requires B, H >= 1, N >= 1, d_v >= 4, d_v % 4 == 0. */
int sdm_fill_state(float* M, float value, int B, int H, long long N, int d_v, void* stream);

/* sdm_select - product-key slot selection ("Meccanismo Core" item 2).
 * For every (b, h, t): halves a = kp[b,h,t,0,:], b = kp[b,h,t,1,:] (S entries each,
 * the sub-scores themselves).  With k = min(W, S), the top-k of each half by
 * (value desc, index asc) are combined into the k x k grid of fp32 sums
 * a[i] + b[j] at flat slot i*S + j, and the top-W of the grid by (sum desc, flat
 * asc) are returned: idx_w[b,h,t,:] (int32 flat slots) and sc_w[b,h,t,:] (fp32
 * sums), best first.  This equals the top-W of all N = S*S slot scores
 * (topk(s1 (+) s2) = topk(topk(s1) (+) topk(s2))).  The same for q' with R.
 *   kp, qp       [B, H, T, 2, S] in_dt (SDM_F32 or SDM_BF16)
 *   idx_w, sc_w  [B, H, T, W] written;  idx_r, sc_r [B, H, T, R] written.
 * Requires 1 <= S <= SDM_MAX_S, 1 <= W, R <= min(S*S, SDM_MAX_K), T >= 0.
 * Results are bit-identical from run to run. */
int sdm_select(const void* kp, const void* qp, int in_dt, int B, int H, int T, int S, int W, int R,
               int32_t* idx_w, float* sc_w, int32_t* idx_r, float* sc_r, void* stream);

/* sdm_select with the kernel chosen (same results, bit for bit, on every path):
 *   path 0  automatic: for bf16 halves with S % 8 == 0, S <= 1024 and W, R <= 128 the
 *           counting selection (one histogram of exact values per half, whose prefix sums
 *           place every selected key; a half or an outer top-K whose largest values do not
 *           fit its 256-bin window falls back to the general steps), else the general one;
 *   path 1  the general selection (radix select on composite keys, then a bitonic sort);
 *   path 2  the counting selection; SDM_EUNSUPPORTED outside its limits (fp32 halves
 *           included).
 * Any other path: SDM_EINVAL.  For tests and measurement. */
int sdm_select_tuned(const void* kp, const void* qp, int in_dt, int B, int H, int T, int S, int W,
                     int R, int32_t* idx_w, float* sc_w, int32_t* idx_r, float* sc_r, int path,
                     void* stream);

/* Bytes of device workspace sdm_scan_forward needs for these sizes (0 when T == 0 or a size
 * is below its minimum; SIZE_MAX when the product does not fit in a size_t). */
size_t sdm_scan_workspace_size(int B, int H, int T, int d_v, int W, int R);

/* sdm_scan_forward - the recurrent sparse gated-delta scan ("Meccanismo Core"
 * items 3 and 4) over T tokens of every (b, h), continuing from the state in M.
 *   M      [B, H, N, d_v] fp32, in: state before token 0, out: state after token T-1.
 *   idx_w, sc_w [B, H, T, W]; idx_r, sc_r [B, H, T, R] as written by sdm_select
 *          (slots distinct within a token's write set).
 *   v      [B, H, T, d_v] v_dt;  alpha, beta [B, H, T] fp32.
 *   o      [B, H, T, d_v] fp32, written: o_t = sum_i softmax(sc_r[t])_i M_t[idx_r[t,i]].
 *   workspace  device scratch of at least sdm_scan_workspace_size(...) bytes, 16-byte
 *          aligned; its contents on entry do not matter and are clobbered.
 *   dev_err  device int, may be NULL; SDM_DEV_* bits are OR-ed in.
 * Calls chained on one stream continue one another exactly: running T1 tokens then
 * T2 tokens gives bit-identical results to one call over T1 + T2 tokens.
 * Requires d_v % 4 == 0, 4 <= d_v <= SDM_MAX_DV, 1 <= W, R <= SDM_MAX_K, N >= max(W, R). */
int sdm_scan_forward(float* M, const int32_t* idx_w, const float* sc_w, const int32_t* idx_r,
                     const float* sc_r, const void* v, int v_dt, const float* alpha,
                     const float* beta, int B, int H, int T, long long N, int d_v, int W, int R,
                     float* o, void* workspace, size_t workspace_bytes, int* dev_err,
                     void* stream);

/* Same as sdm_scan_forward with the scan kernel's shape forced instead of chosen:
 * cols_per_cta in {4, 8, 16, 32, 64} (d_v columns owned by one thread block,
 * d_v % cols == 0) and prefetch_depth in {1, 2, 3} (tokens of rows gathered ahead; 64
 * columns allow 1 or 2).  0 keeps the automatic choice.  The state and the slots do not
 * depend on the shape; o may differ in the last bits (order of the read reduction).
 * `wait_before_scan`, if not NULL, is a cudaEvent_t the stream waits for after the
 * planning kernel (which does not read M) and before the scan kernel: M only has to be
 * ready then, so work producing M (e.g. sdm_init_state_from_M0 on another stream) can
 * overlap the selection and planning.  `event_after_plan`, if not NULL, is a cudaEvent_t
 * recorded on `stream` right before the scan kernel (after that wait), for timing the
 * scan kernel alone.  For tuning, tests, measurement and stream-level overlap. */
int sdm_scan_forward_tuned(float* M, const int32_t* idx_w, const float* sc_w,
                           const int32_t* idx_r, const float* sc_r, const void* v, int v_dt,
                           const float* alpha, const float* beta, int B, int H, int T,
                           long long N, int d_v, int W, int R, float* o, void* workspace,
                           size_t workspace_bytes, int* dev_err, int cols_per_cta,
                           int prefetch_depth, void* event_after_plan, void* wait_before_scan,
                           void* stream);

/* Bytes of the fixed device scratch behind sdm_scan_forward_noalloc (64 MiB). */
#define SDM_NOALLOC_SCRATCH_BYTES (64u << 20)

/* sdm_scan_forward_noalloc - sdm_scan_forward without a caller-provided workspace; the
 * paper has no counterpart: this is an interface for callers that cannot allocate device
 * memory where they run the scan (a serving or real-time loop that forbids allocation on
 * its request path, or a host application that owns no allocator and passes only its
 * input and output buffers).  Same arguments, results and errors as sdm_scan_forward,
 * minus the workspace; the library calls no cudaMalloc/cudaFree or other allocating
 * routine for it.  The host checks run in this order, before anything is launched: the
 * argument checks of sdm_scan_forward (SDM_EINVAL, SDM_EUNSUPPORTED, SDM_EALIGN), then a
 * workspace size that does not fit in a size_t (SDM_EUNSUPPORTED), then the scratch
 * size (SDM_ESCRATCH).
 *   - The planning records go to one fixed scratch of SDM_NOALLOC_SCRATCH_BYTES that lives
 *     in the library's device image: every GPU that loads the library keeps that memory
 *     until the process exits.
 *   - Sizes whose workspace (sdm_scan_workspace_size) exceeds SDM_NOALLOC_SCRATCH_BYTES are
 *     refused with SDM_ESCRATCH before anything is launched; e.g. with d_v = 128 and
 *     W = R = 128 (3,088 bytes per (b, h, t)) up to 21,732 (b, h, t) triples per call.
 *   - The first call on a device looks up the scratch's device address (once per device,
 *     with that device current); make that first call before any stream capture.  The
 *     address is kept for the life of the process: after a cudaDeviceReset of a device
 *     the library's device image is loaded anew, so do not call this entry point on that
 *     device again in the same process.
 *   - All calls on a device share the scratch and each one overwrites what the last left
 *     there (nothing in it needs to start at zero).  Calls whose work overlaps on the GPU
 *     (other streams, other host threads) race on it: keep them ordered, e.g. on one
 *     stream. */
int sdm_scan_forward_noalloc(float* M, const int32_t* idx_w, const float* sc_w,
                             const int32_t* idx_r, const float* sc_r, const void* v, int v_dt,
                             const float* alpha, const float* beta, int B, int H, int T,
                             long long N, int d_v, int W, int R, float* o, int* dev_err,
                             void* stream);

/* The scan kernel shape sdm_scan_forward would use (host-only query): columns per
 * thread block, prefetch depth, thread blocks, dynamic shared memory bytes. */
int sdm_scan_launch_info(int B, int H, int d_v, int W, int R, int* cols_per_cta,
                         int* prefetch_depth, int* blocks, int* smem_bytes);

/* sdm_forward - one whole forward pass of the SDM layer over a batch of sequences
 * ("Stato Iniziale Appreso": every sequence starts from the learned M_0; "Meccanismo
 * Core" items 2-4: product-key selection, gated delta write, read after write), with
 * the selection and the scan overlapped in token chunks on internal streams.  Results
 * are bit-identical to sdm_init_state_from_M0 + sdm_select + sdm_scan_forward on one
 * stream.
 *   kp, qp [B, H, T, 2, S] in_dt; v [B, H, T, d_v] v_dt; alpha, beta [B, H, T] fp32.
 *   M0     [H, N, d_v] fp32 with N = S*S, or NULL to continue from the state in M.
 *   M      [B, H, N, d_v] fp32, out: state after token T-1.
 *   idx_w, sc_w [B, H, T, W]; idx_r, sc_r [B, H, T, R]; o [B, H, T, d_v] fp32: written,
 *          as by sdm_select and sdm_scan_forward.
 *   workspace  device scratch of at least sdm_forward_workspace_size(B, H, T, d_v, W, R, 0)
 *          bytes, 16-byte aligned, contents irrelevant.
 *   dev_err  device int or NULL, as for sdm_scan_forward.
 * Ordering: work enqueued on `stream` before the call runs before any of the call's work,
 * and work enqueued on `stream` after the call sees all of its results.  The library
 * runs the work on four streams of its own per device (created on the first call on
 * that device) and enqueues calls on one device one at a time.  Concurrent calls that
 * share M, the outputs or the workspace race, as with any of these entry points.
 * Errors: the argument checks of sdm_select and sdm_scan_forward (nothing enqueued);
 * SDM_ENOSPACE for a short workspace; SDM_ECUDA if a launch fails part-way, after
 * which M and the outputs are unspecified. */
size_t sdm_forward_workspace_size(int B, int H, int T, int d_v, int W, int R, int chunks);
int sdm_forward(const void* kp, const void* qp, int in_dt, const void* v, int v_dt,
                const float* alpha, const float* beta, const float* M0, float* M, int B, int H,
                int T, int S, int d_v, int W, int R, int32_t* idx_w, float* sc_w, int32_t* idx_r,
                float* sc_r, float* o, void* workspace, size_t workspace_bytes, int* dev_err,
                void* stream);

/* sdm_forward with the chunking chosen: `chunks` token chunks (0 = automatic: about 512
 * tokens each, 1024 when T >= 8192; the effective count is sdm_forward_chunks(T, chunks)),
 * and, when
 * `scan_events` is not NULL, 2 * chunks cudaEvent_t recorded right before and after each
 * chunk's scan kernel on the stream it runs on (for timing the scan kernel).  The
 * workspace must hold sdm_forward_workspace_size(..., chunks) bytes. */
int sdm_forward_chunks(int T, int chunks);
/* sdm_forward_tuned whose inputs may still be arriving: when `input_ready` is not NULL it
 * holds sdm_forward_chunks(T, chunks) cudaEvent_t (an entry may be NULL), and the selection
 * and planning of token chunk c (tokens c*Tc .. c*Tc+Tc-1 of every (b, h), Tc =
 * ceil(T / chunks)) start only after input_ready[c] (its latest record at the time of the
 * call) has completed; the state initialisation does not wait.  So a caller copying a
 * batch's inputs token window by token window (sdm_copy_rows_async) lets the pass start on
 * the first window.  The events are only waited on, never recorded; the rest is
 * sdm_forward_tuned. */
int sdm_forward_streamed(const void* kp, const void* qp, int in_dt, const void* v, int v_dt,
                         const float* alpha, const float* beta, const float* M0, float* M, int B,
                         int H, int T, int S, int d_v, int W, int R, int32_t* idx_w, float* sc_w,
                         int32_t* idx_r, float* sc_r, float* o, void* workspace,
                         size_t workspace_bytes, int* dev_err, int chunks,
                         void* const* scan_events, void* const* input_ready, void* stream);
/* sdm_copy_rows_async - `rows` rows of `row_bytes` bytes from src (rows `src_pitch` bytes
 * apart) to dst (rows `dst_pitch` bytes apart), asynchronously on `stream`; either side may
 * be device memory or pinned host memory (the direction follows from the addresses).  One
 * token window of a [B, H, T, ...] input for every (b, h) is B*H such rows.  SDM_EINVAL for
 * null pointers or a pitch below row_bytes; nothing to do for zero rows or bytes. */
int sdm_copy_rows_async(void* dst, size_t dst_pitch, const void* src, size_t src_pitch,
                        size_t row_bytes, size_t rows, void* stream);
int sdm_forward_tuned(const void* kp, const void* qp, int in_dt, const void* v, int v_dt,
                      const float* alpha, const float* beta, const float* M0, float* M, int B,
                      int H, int T, int S, int d_v, int W, int R, int32_t* idx_w, float* sc_w,
                      int32_t* idx_r, float* sc_r, float* o, void* workspace,
                      size_t workspace_bytes, int* dev_err, int chunks, void* const* scan_events,
                      void* stream);

/* Backward pass (training) of the scan, for the loss L = sum_t <dO_t, o_t> + <dM_T, M_T>
 * with the selected slots held fixed (they are discrete); gradients reach v, alpha, beta,
 * the selected write and read scores, the initial state ("Stato Iniziale Appreso": M_0 is
 * learned) and, through sdm_select_backward, the k' / q' halves ("Meccanismo Core" item 2:
 * a selected score is half0[i] + half1[j]).
 *
 * sdm_scan_forward_train - sdm_scan_forward that also stores what the backward needs:
 *   w_prev [B, H, T, W, d_v] fp32: every write row before its update (M_{t-1}[idx_w]);
 *   r_rows [B, H, T, R, d_v] fp32: every read row as read (M_t[idx_r]).
 * Rows of invalid slots (dev_err SDM_DEV_INDEX_RANGE) are not stored. */
int sdm_scan_forward_train(float* M, const int32_t* idx_w, const float* sc_w,
                           const int32_t* idx_r, const float* sc_r, const void* v, int v_dt,
                           const float* alpha, const float* beta, int B, int H, int T,
                           long long N, int d_v, int W, int R, float* o, float* w_prev,
                           float* r_rows, void* workspace, size_t workspace_bytes, int* dev_err,
                           void* stream);

/* sdm_scan_backward - the reverse-mode pass.
 *   idx/sc, v, alpha, beta: as given to sdm_scan_forward_train; w_prev, r_rows: its outputs.
 *   dO     [B, H, T, d_v] fp32: dL/do.
 *   G      [B, H, N, d_v] fp32, in: dL/dM_T (zeros when the final state carries no
 *          gradient), out: dL/dM_0 for each (b, h) (overwritten in place).
 *   dv     [B, H, T, d_v] fp32; dalpha, dbeta [B, H, T]; dsc_w [B, H, T, W];
 *          dsc_r [B, H, T, R]: written.
 *   dM0    [H, N, d_v] fp32 or NULL: if given, the sum of the output G over the batch
 *          (the gradient of an M_0 shared by the batch).
 *   workspace  at least sdm_scan_backward_workspace_size(...) bytes, 16-byte aligned,
 *          contents irrelevant (per (b, h, t): the column slices' partial sums and the
 *          softmax weights of the token's scores, formed by a parallel pass first).
 * Requires d_v % 4 == 0 and the limits of sdm_scan_forward; slots outside [0, N) are
 * skipped (their gradients are unspecified).  A token's write slots are distinct, and so
 * are its read slots (as sdm_select gives them); a repeated slot within either set gives
 * unspecified gradients. */
size_t sdm_scan_backward_workspace_size(int B, int H, int T, int d_v, int W, int R);

/* sdm_scan_backward_ex - sdm_scan_backward with flags (0: the same call).
 *   SDM_BWD_FINAL_ZERO: dL/dM_T is zero (the loss reads the outputs only).  G's contents on
 *          entry are ignored (it need not be cleared); on exit it holds dL/dM_0 for each
 *          (b, h) as without the flag, with G cleared: exactly equal values (a zero's sign
 *          may differ).  Knowing that the adjoint starts at zero, the pass finds, per slot,
 *          whether the adjoint row there is still zero (no later read selects the row) and
 *          skips that row's loads and, for a write slot, its store.  Three more kernels
 *          (the last token reading each row, one bit per slot) run first; with T = 0 every
 *          row of G is set to zero.
 *   workspace  at least sdm_scan_backward_workspace_size_ex(B, H, T, N, d_v, W, R, flags)
 *          bytes (with the flag: 4 bytes per (b, h, row) and 4 per 32 slots of a token more),
 *          16-byte aligned, contents irrelevant.
 * Unknown flag bits: SDM_EINVAL (and a workspace size of 0).  Two read slots of one token
 * naming the same row give unspecified gradients, as in sdm_scan_backward. */
#define SDM_BWD_FINAL_ZERO 1u
/*   SDM_BWD_DM0_ONLY (with SDM_BWD_FINAL_ZERO): the caller needs the batch's dM0 but not G
 *          per (b, h): the rows of G that no slot reads are left as they were instead of
 *          being set to zero (G's contents on exit unspecified; dM0 and the other outputs
 *          are those of the call without the flag).  dM0 must not be NULL (SDM_EINVAL).
 *          Without SDM_BWD_FINAL_ZERO the flag changes nothing. */
#define SDM_BWD_DM0_ONLY 2u
size_t sdm_scan_backward_workspace_size_ex(int B, int H, int T, long long N, int d_v, int W, int R,
                                           unsigned flags);
int sdm_scan_backward_ex(const int32_t* idx_w, const float* sc_w, const int32_t* idx_r,
                         const float* sc_r, const void* v, int v_dt, const float* alpha,
                         const float* beta, const float* w_prev, const float* r_rows,
                         const float* dO, int B, int H, int T, long long N, int d_v, int W, int R,
                         float* G, float* dv, float* dalpha, float* dbeta, float* dsc_w,
                         float* dsc_r, float* dM0, unsigned flags, void* workspace,
                         size_t workspace_bytes, void* stream);
int sdm_scan_backward(const int32_t* idx_w, const float* sc_w, const int32_t* idx_r,
                      const float* sc_r, const void* v, int v_dt, const float* alpha,
                      const float* beta, const float* w_prev, const float* r_rows,
                      const float* dO, int B, int H, int T, long long N, int d_v, int W, int R,
                      float* G, float* dv, float* dalpha, float* dbeta, float* dsc_w,
                      float* dsc_r, float* dM0, void* workspace, size_t workspace_bytes,
                      void* stream);

/* sdm_select_backward - gradient of the selected scores with respect to the halves:
 * dhalves[b, h, t, 0, i] = sum of dsc over the selected slots with flat / S == i, and
 * dhalves[b, h, t, 1, j] over those with flat % S == j.  idx, dsc [B, H, T, K] (as from
 * sdm_select and sdm_scan_backward); dhalves [B, H, T, 2, S] fp32, overwritten.  The sums
 * use atomic adds: their order, and so the last bits, may vary from run to run. */
int sdm_select_backward(const int32_t* idx, const float* dsc, int B, int H, int T, int S, int K,
                        float* dhalves, void* stream);

/* sdm_decode_step - one decode token (T = 1) for every (b, h), in a single kernel: the
 * selection of sdm_select, then the gated delta write and the read of sdm_scan_forward,
 * with the state resident in M ("Meccanismo Core" items 2-4 applied to one token).
 * Arguments as for sdm_select and sdm_scan_forward with T = 1 (kp, qp [B, H, 1, 2, S];
 * v [B, H, 1, d_v]; alpha, beta [B, H, 1]; idx/sc [B, H, 1, W or R]; o [B, H, 1, d_v]);
 * no workspace.  Every output (slots, scores, o, M) is bit-identical to sdm_select followed
 * by sdm_scan_forward over the same token: a block covers the column slice the scan
 * kernel would use for these sizes, so the read is summed in the same order.
 * SDM_EUNSUPPORTED when the block's shared memory would not fit (very large W + R or S);
 * sdm_decode_step_supported answers that on the host (SDM_OK or SDM_EUNSUPPORTED). */
int sdm_decode_step(const void* kp, const void* qp, int in_dt, const void* v, int v_dt,
                    const float* alpha, const float* beta, float* M, int B, int H, int S, int d_v,
                    int W, int R, int32_t* idx_w, float* sc_w, int32_t* idx_r, float* sc_r,
                    float* o, int* dev_err, void* stream);
int sdm_decode_step_supported(int in_dt, int B, int H, int S, int d_v, int W, int R);

/* The staircase table of a decode step: for the write task and then the read task, the pairs
 * (p, q) of ranks in the two sorted inner top-k lists whose rank product (p+1)(q+1) is at most
 * K (W or R), the only pairs that can hold one of the K largest sums ("Meccanismo Core" item
 * 2).  It depends on W, R and S alone, so a caller stepping one shape token after token builds
 * it once and passes it to every step instead of each step's blocks building it.
 * sdm_decode_table_words - its size in 32-bit words (-1 for sizes sdm_decode_step rejects).
 * sdm_decode_table - writes it into `table` (caller-owned device memory of at least that many
 *   words, 4-byte aligned) on `stream`.  SDM_EINVAL for a null table or rejected sizes.
 * sdm_decode_step_tabled - sdm_decode_step whose blocks read the staircases from `table` (as
 *   written by sdm_decode_table for the same W, R and S, and not written while the step runs;
 *   NULL: the blocks build them, as sdm_decode_step does).  The same bits either way. */
int sdm_decode_table_words(int W, int R, int S);
int sdm_decode_table(uint32_t* table, int W, int R, int S, void* stream);
int sdm_decode_step_tabled(const void* kp, const void* qp, int in_dt, const void* v, int v_dt,
                           const float* alpha, const float* beta, float* M, int B, int H, int S,
                           int d_v, int W, int R, int32_t* idx_w, float* sc_w, int32_t* idx_r,
                           float* sc_r, float* o, int* dev_err, const uint32_t* table,
                           void* stream);

/* sdm_project_kq - the projections that produce the product keys and queries
 * ("Meccanismo Core" item 2: the projected key k' and query q', whose two halves are the
 * sub-scores; "Design IsoFLOP": the projections are linear layers).  One bf16 GEMM on the
 * tensor cores (fp32 accumulation, each output rounded to bf16, nearest even):
 *   kp[b,h,t,half,s] = sum_d x[b,t,d] * w[(h*2 + half)*S + s, d]
 *   qp[b,h,t,half,s] = sum_d x[b,t,d] * w[H*2*S + (h*2 + half)*S + s, d]
 *   x  [B, T, D] bf16 (raw 16-bit patterns), read only;
 *   w  [4*H*S, D] bf16, read only: one row of D weights per output column, the k'
 *      columns (head, half, index) first, then the q' columns in the same order;
 *   kp, qp [B, H, T, 2, S] bf16, written (the layout sdm_select reads, in_dt SDM_BF16).
 * The order of the fp32 accumulation is unspecified, so an output can differ from the
 * correctly rounded sum by one bf16 unit where the sum lies near a rounding boundary.
 * Requires B, T, H >= 1, 1 <= S <= SDM_MAX_S, D >= 8 with D % 8 == 0 (the row pitch of x
 * and w is a multiple of 16 bytes), B*T < 2^31, 4*H*S < 2^31; x, w, kp, qp 16-byte
 * aligned.  dev_err: device int or NULL; SDM_DEV_TIMEOUT if a wait inside the kernel ran
 * out (then kp, qp are unspecified).  Runs as one persistent kernel on `stream`: one
 * block per SM, in clusters of two blocks that compute 256 x 256 output tiles together. */
int sdm_project_kq(const void* x, const void* w, int B, int T, int D, int H, int S, void* kp,
                   void* qp, int* dev_err, void* stream);

/* sdm_project_kq_tuned - sdm_project_kq with its launch shape fixed by the caller:
 *   max_ctas  at most this many blocks (0: as many as can be resident, one per SM), to leave
 *             SMs to work running beside it on other streams;
 *   pair      2: clusters of two blocks whose MMAs run as one 256-row tile across both SMs
 *             (tcgen05 cta_group::2), each block staging its own rows of x and half of the
 *             weight tile; 0: single blocks (128 x 256 tiles); -1: 2 unless B*T <= 128
 *             (then 0).  Any other value: SDM_EINVAL.
 * Results do not depend on either. */
int sdm_project_kq_tuned(const void* x, const void* w, int B, int T, int D, int H, int S,
                         void* kp, void* qp, int* dev_err, int max_ctas, int pair, void* stream);

/* sdm_project_select - the projections fused with the selection ("Meccanismo Core" item 2:
 * the projected k' and q', whose halves are the sub-scores, and the top-k of each half;
 * "Design IsoFLOP": the projections are linear layers).  The same results as
 * sdm_project_kq followed by sdm_select on its output, bit for bit, without k' and q' ever
 * being written to device memory: one kernel computes the projections on the tensor cores
 * (tcgen05, fp32 accumulation in the same order as sdm_project_kq) and, on chip, rounds each
 * half to bf16 and takes its top-min(K, S) by (value desc, index asc); a second kernel takes
 * the outer top-K over each task's two lists.
 *   x  [B, T, D] bf16, w [4*H*S, D] bf16: as for sdm_project_kq;
 *   idx_w, sc_w [B, H, T, W]; idx_r, sc_r [B, H, T, R]: written, as by sdm_select.
 *   workspace  device scratch of at least sdm_project_select_workspace_size(B, T, H, S, W, R)
 *          bytes (the per-half lists, 4 bytes per entry, and the staircase table), 16-byte
 *          aligned, contents irrelevant.
 *   dev_err  device int or NULL: SDM_DEV_TIMEOUT if a wait inside the kernel ran out.
 * Requires the limits of sdm_project_kq and, for this kernel, S % 128 == 0, S <= 1024 and
 * W, R <= 128 (SDM_EUNSUPPORTED otherwise); SDM_ENOSPACE for a short workspace. */
size_t sdm_project_select_workspace_size(int B, int T, int H, int S, int W, int R);
int sdm_project_select(const void* x, const void* w, int B, int T, int D, int H, int S, int W,
                       int R, int32_t* idx_w, float* sc_w, int32_t* idx_r, float* sc_r,
                       void* workspace, size_t workspace_bytes, int* dev_err, void* stream);

/* sdm_test_bounded_wait - test of the timeout path of the projection kernel's waits (not
 * part of the method): one warp waits once, with the same bounded mbarrier wait, on a
 * barrier of its own:
 *   mode 0  on a phase that nothing completes: the wait gives up after limit_ns;
 *   mode 1  on a phase already completed by its own arrival: returns at once;
 *   mode 2  with the block's stop flag already raised: gives up at once.
 * When the wait gave up, SDM_DEV_TIMEOUT is OR-ed into *dev_err (device int, required), as
 * the projection kernel does.  elapsed_ns (device, 8-byte aligned, or NULL) receives the
 * wait's duration from the global timer.  limit_ns <= 10^9; SDM_EINVAL otherwise.  The
 * kernel issues no copies, so nothing is left in flight and the context stays usable. */
int sdm_test_bounded_wait(int mode, unsigned long long limit_ns, int* dev_err,
                          unsigned long long* elapsed_ns, void* stream);

/* sdm_test_project_stall - test of the projection kernel's stop and drain path (not part of
 * the method): sdm_project_kq_tuned(..., max_ctas 0, pair) in which the copy-issuing thread
 * of cluster rank stall_cta (0 or, with pair 2, 1) stops issuing after stall_step K steps,
 * as if its copies could not be issued, and every wait inside the kernel gives up after
 * wait_ns.  The waits for the missing copies then run out, the blocks stop, wait for every
 * copy they (and, in a pair, the peer block) issued to land, free their tensor memory and
 * OR SDM_DEV_TIMEOUT into *dev_err (device int, required); kp, qp are unspecified.  With
 * pair 2 one rank's producer runs ahead of the other's, so the pair's drain meets phases
 * only one of them issued.  Requires the arguments of sdm_project_kq, pair 0 or 2 (2: B*T >
 * 128), 10^5 <= wait_ns <= 10^9 (SDM_EINVAL otherwise).  Nothing waits longer than wait_ns
 * for something that cannot happen, so the call returns and the context stays usable. */
int sdm_test_project_stall(const void* x, const void* w, int B, int T, int D, int H, int S,
                           void* kp, void* qp, int pair, int stall_cta, int stall_step,
                           unsigned long long wait_ns, int* dev_err, void* stream);

/* sdm_gen_inputs - synthetic inputs (not part of the method): draws the box
 * b in [b_off, b_off+B), all H heads, tokens t in [t_off, t_off+T) of a logical
 * workload with T_total tokens per sequence, from the counter-based generator
 * (Philox4x32-10 keyed by `seed`, Box-Muller with fixed fp32 series; bit-identical
 * to the host generator that feeds the CPU reference).
 *   kp, qp [B, H, T, 2, S] in_dt: N(0,1) (+ half_bias[j] on index j of every half
 *          when half_bias, a device fp32 [S] array, is not NULL);
 *   v [B, H, T, d_v] in_dt: N(0,1);  alpha [B, H, T] fp32: U(alpha_lo, 1);
 *   beta [B, H, T] fp32: U(0, 1) if beta_kind == 0, sigmoid(N(0,1)) if 1.
 * Any of kp, qp, v, alpha, beta may be NULL to skip that tensor. */
int sdm_gen_inputs(unsigned long long seed, int B, int H, int T, int b_off, int t_off,
                   long long T_total, int S, int d_v, int in_dt, float alpha_lo, int beta_kind,
                   const float* half_bias, void* kp, void* qp, void* v, float* alpha,
                   float* beta, void* stream);

/* sdm_gen_M0 - synthetic learned initial state: M0 [H, N, d_v] fp32 = scale * N(0,1)
 * from the same generator (field of M_0). */
int sdm_gen_M0(unsigned long long seed, int H, long long N, int d_v, float scale, float* M0,
               void* stream);

#ifdef __cplusplus
}
#endif

#endif /* SDM_H_ */
