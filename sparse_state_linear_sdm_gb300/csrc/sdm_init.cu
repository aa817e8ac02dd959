// State initialisation from the learned initial state (Sparse Delta Memory technical
// summary, gist.science/it/paper/2607.07386, "Stato Iniziale Appreso": M_0 is a
// learnable parameter that every sequence starts from).
// M[b, h] = M0[h]: each 16-byte chunk of M0 is read once and stored B times, so the
// HBM traffic is exactly |M0| read + |M| written.  Pure bandwidth.
//
// The kernel is meant to run beside the selection kernel (another stream), so it takes
// little of each SM: one block per SM (which already saturates HBM writes), and the
// SM's shared memory left at its maximum split, so that selection blocks (tens of KB
// of shared memory each) can start on the same SM without waiting for it to drain.
//
// The pipelined pass does not copy M_0 up front.  A row keeps M_0's value until the first
// token that writes it, so it is enough to know, per slot, the first token that writes it
// (launch_first_writes, one atomic minimum per selected write slot): the planning pass
// sends gathers of rows not yet written to M_0, and launch_fill_unwritten copies M_0 into
// the rows that no token writes, once the last chunk's slots are known.  The copy and the
// scans touch disjoint rows, so they can run at the same time.
#include "sdm_internal.cuh"

namespace sdm {
namespace {

__global__ void __launch_bounds__(256) init_state_kernel(float4* __restrict__ M,
                                                         const float4* __restrict__ M0, int B,
                                                         size_t per_batch4) {
  const size_t stride = size_t(gridDim.x) * blockDim.x;
  for (size_t i = size_t(blockIdx.x) * blockDim.x + threadIdx.x; i < per_batch4; i += stride) {
    const float4 x = __ldcs(M0 + i);
    for (int b = 0; b < B; ++b) __stcs(M + size_t(b) * per_batch4 + i, x);
  }
}

__global__ void __launch_bounds__(256) first_writes_kernel(const int32_t* __restrict__ idx_w,
                                                           int32_t* __restrict__ first, int BH,
                                                           int Tc, int T_total, int t0, int W,
                                                           long long N) {
  const size_t per_bh = size_t(Tc) * W;
  const size_t total = size_t(BH) * per_bh;
  const size_t stride = size_t(gridDim.x) * blockDim.x;
  for (size_t i = size_t(blockIdx.x) * blockDim.x + threadIdx.x; i < total; i += stride) {
    const size_t bh = i / per_bh, rem = i - bh * per_bh;
    const int32_t x = idx_w[(bh * T_total + t0) * W + rem];
    if (x < 0 || x >= N) continue;
    atomicMin(first + bh * size_t(N) + size_t(x), t0 + int(rem / W));
  }
}

// One warp per (head h, row x): lane l reads the first-write entry of sequence b = l (32
// sequences per round), a ballot gives the sequences whose row x was never written, and the
// M_0 row, loaded once, is stored into each of them.  Consecutive warps take consecutive
// rows, so the entries of neighbouring rows share sectors in L2.
__global__ void __launch_bounds__(256) fill_unwritten_kernel(float* __restrict__ M,
                                                             const float* __restrict__ M0,
                                                             const int32_t* __restrict__ first,
                                                             int B, int H, long long N, int d_v) {
  const int lane = threadIdx.x & 31;
  const long long items = (long long)H * N;
  const long long warps = (long long)gridDim.x * (blockDim.x / 32);
  const int q4 = d_v / 4;
  for (long long it = (long long)blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5); it < items;
       it += warps) {
    const int h = int(it / N);
    const long long x = it - (long long)h * N;
    const float4* src = reinterpret_cast<const float4*>(M0 + size_t(it) * d_v);
    for (int b0 = 0; b0 < B; b0 += 32) {
      const int b = b0 + lane;
      const bool mine = b < B && first[(size_t(b) * H + h) * size_t(N) + size_t(x)] == kNeverWritten;
      const unsigned need = __ballot_sync(0xFFFFFFFFu, mine);
      if (!need) continue;
      for (int k = lane; k < q4; k += 32) {
        const float4 val = __ldg(src + k);
        for (unsigned m = need; m; m &= m - 1) {
          const size_t bh = size_t(b0 + __ffs(m) - 1) * H + h;
          __stcs(reinterpret_cast<float4*>(M + (bh * size_t(N) + size_t(x)) * d_v) + k, val);
        }
      }
    }
  }
}

int sm_count_now() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return -1;
  return sms;
}

}  // namespace

int launch_first_writes(const int32_t* idx_w, const TokenWindow& win, long long N, int W,
                        int32_t* first_write, cudaStream_t s) {
  const size_t total = size_t(win.BH) * size_t(win.Tc) * size_t(W);
  if (total == 0) return SDM_OK;
  const int sms = sm_count_now();
  if (sms <= 0) return SDM_ECUDA;
  size_t blocks = size_t(sms) * 4;
  const size_t need = (total + 255) / 256;
  if (blocks > need) blocks = need;
  first_writes_kernel<<<unsigned(blocks), 256, 0, s>>>(idx_w, first_write, win.BH, win.Tc,
                                                        win.T_total, win.t0, W, N);
  return last_launch_status();
}

int launch_fill_unwritten(float* M, const float* M0, const int32_t* first_write, int B, int H,
                          long long N, int d_v, cudaStream_t s) {
  if (B == 0 || H == 0 || N == 0) return SDM_OK;
  const int sms = sm_count_now();
  if (sms <= 0) return SDM_ECUDA;
  if (cudaFuncSetAttribute(reinterpret_cast<const void*>(&fill_unwritten_kernel),
                           cudaFuncAttributePreferredSharedMemoryCarveout,
                           int(cudaSharedmemCarveoutMaxShared)) != cudaSuccess)
    return SDM_ECUDA;
  const long long items = (long long)H * N;
  long long blocks = (long long)sms * 8;
  if (blocks > (items + 7) / 8) blocks = (items + 7) / 8;
  fill_unwritten_kernel<<<unsigned(blocks), 256, 0, s>>>(M, M0, first_write, B, H, N, d_v);
  return last_launch_status();
}

int launch_init_state(float* M, const float* M0, int B, int H, long long N, int d_v,
                      cudaStream_t s) {
  const size_t per_batch4 = size_t(H) * size_t(N) * size_t(d_v) / 4;
  if (per_batch4 == 0) return SDM_OK;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return SDM_ECUDA;
  if (cudaFuncSetAttribute(reinterpret_cast<const void*>(&init_state_kernel),
                           cudaFuncAttributePreferredSharedMemoryCarveout,
                           int(cudaSharedmemCarveoutMaxShared)) != cudaSuccess)
    return SDM_ECUDA;
  size_t blocks = size_t(sms);
  const size_t need = (per_batch4 + 255) / 256;
  if (blocks > need) blocks = need;
  init_state_kernel<<<unsigned(blocks), 256, 0, s>>>(reinterpret_cast<float4*>(M),
                                                     reinterpret_cast<const float4*>(M0), B,
                                                     per_batch4);
  return last_launch_status();
}

}  // namespace sdm
