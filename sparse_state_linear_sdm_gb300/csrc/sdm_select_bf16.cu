// Product-key selection for bf16 sub-scores: the counting selection (sdm_select_count.cuh)
// where its limits hold, else the general kernels (sdm_select_impl.cuh).
#include "sdm_select_count.cuh"

namespace sdm {
int launch_select_bf16(const void* kp, const void* qp, const TokenWindow& win, int S, int W, int R,
                       int32_t* idx_w, float* sc_w, int32_t* idx_r, float* sc_r, cudaStream_t s,
                       const uint32_t* stair_g, int path) {
  if (path != kSelectGeneral) {
    const int st = launch_select_count(kp, qp, win, S, W, R, idx_w, sc_w, idx_r, sc_r, s, stair_g,
                                       path == kSelectCounting);
    if (st != SDM_EUNSUPPORTED || path == kSelectCounting) return st;
  }
  return launch_select_t<uint16_t>(kp, qp, win, S, W, R, idx_w, sc_w, idx_r, sc_r, s, stair_g);
}

// The write and read staircases of a (W, R, S) selection as one table in device memory,
// built once by one block so that the selection blocks of a pipelined forward pass read it
// instead of each building its own.
int stair_table_words(int W, int R, int S) {
  return stair_count(W, min(W, S)) + stair_count(R, min(R, S));
}
int launch_stair_table(uint32_t* out, int W, int R, int S, cudaStream_t s) {
  stair_table_kernel<<<1, 128, 0, s>>>(out, W, R, S);
  return last_launch_status();
}
}  // namespace sdm
