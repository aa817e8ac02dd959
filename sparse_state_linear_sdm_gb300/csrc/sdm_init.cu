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

// Every float of a state-shaped table set to `value` (streaming stores, 16 bytes a thread).
__global__ void __launch_bounds__(256) fill_state_kernel(float4* __restrict__ M, float value,
                                                         size_t n4) {
  const size_t stride = size_t(gridDim.x) * blockDim.x;
  const float4 x = make_float4(value, value, value, value);
  for (size_t i = size_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n4; i += stride) __stcs(M + i, x);
}

__global__ void __launch_bounds__(256) fill_words_kernel(int32_t* __restrict__ p, int32_t value,
                                                         size_t n) {
  const size_t stride = size_t(gridDim.x) * blockDim.x;
  for (size_t i = size_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride) p[i] = value;
}

int grid_cap(size_t work, int per_block) {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return -1;
  size_t blocks = (work + per_block - 1) / per_block;
  const size_t cap = size_t(sms) * 8;
  return int(blocks < cap ? (blocks < 1 ? 1 : blocks) : cap);
}

}  // namespace

int launch_fill_words(int32_t* p, int32_t value, size_t n, cudaStream_t s) {
  if (n == 0) return SDM_OK;
  const int blocks = grid_cap(n, 256);
  if (blocks < 1) return SDM_ECUDA;
  fill_words_kernel<<<blocks, 256, 0, s>>>(p, value, n);
  return last_launch_status();
}

int launch_fill_state(float* M, float value, int B, int H, long long N, int d_v, cudaStream_t s) {
  const size_t n4 = size_t(B) * size_t(H) * size_t(N) * size_t(d_v) / 4;
  if (n4 == 0) return SDM_OK;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return SDM_ECUDA;
  size_t blocks = size_t(sms) * 16;
  const size_t need = (n4 + 255) / 256;
  if (blocks > need) blocks = need;
  fill_state_kernel<<<unsigned(blocks), 256, 0, s>>>(reinterpret_cast<float4*>(M), value, n4);
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
