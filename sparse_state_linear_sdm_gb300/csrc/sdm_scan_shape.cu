// Launch shape of the scan kernel (host side): the column slice per block and the number of
// tokens of rows in flight, from the sizes and this GPU's SM count and shared memory.  Kept
// apart from the kernel's source: the choice is measured per shape, the kernel is not
// touched by it.
#include "sdm_internal.cuh"

namespace sdm {

int choose_scan_shape(int BH, int d_v, int W, int R, int force_cols, int force_pd,
                      ScanShape* out) {
  int dev = 0, max_smem = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return SDM_ECUDA;
  const int col_opts[5] = {64, 32, 16, 8, 4};
  int best_cols = 0, best_pd = 0;
  for (int ci = force_cols ? 0 : 1; ci < 5 && !best_cols; ++ci) {
    const int c = col_opts[ci];
    if (force_cols && c != force_cols) continue;
    if (d_v % c) continue;
    // The widest row slice (up to 128 bytes) that still gives at least 0.8 blocks per SM:
    // a block's chain of tokens is latency-bound, so more chains beat wider rows once the
    // GPU is short of blocks (measured on four shapes: B16 H4 d_v=128 and B8 H16 d_v=64 take
    // 32 columns; B4 H8 d_v=64, 16 columns: 1.75 ms against 1.87 ms with 8; B1 H4 d_v=128, 4
    // columns: 0.93 against 0.99-1.72 us per token with 8-32).
    if (!force_cols && ci + 1 < 5 && d_v % col_opts[ci + 1] == 0 &&
        (long long)BH * (d_v / c) * 5 < 4LL * sms)
      continue;
    // One token of rows in flight per block measured fastest when the blocks fill the GPU
    // (pd 1: 18.8 ms, pd 2: 19.1 ms on B16 H4 T8192 N=2^20 d_v=128 W=R=128) and for short
    // tokens (B4 H8 W=R=32, 128 blocks: 1.75 against 1.86 ms); with fewer blocks than SMs
    // and many rows per token each block's gathers set the pace, and two tokens in flight
    // measured faster (B1 H4 N=2^20 W=R=128, 128 blocks of 4 columns: 0.86 us per token
    // against 0.95 with one token and 0.93 with three; 8 columns 0.94-0.98, 16 columns 1.31).
    const int pd0 = (long long)BH * (d_v / c) < sms && W + R >= 128 ? 2 : 1;
    const int pds[2] = {pd0, 3 - pd0};
    for (int k = 0; k < 2 && !best_cols; ++k) {
      const int p = force_pd ? force_pd : pds[k];
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

}  // namespace sdm
