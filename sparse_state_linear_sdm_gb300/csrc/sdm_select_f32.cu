// Product-key selection for fp32 sub-scores (kernels in sdm_select_impl.cuh).
#include "sdm_select_impl.cuh"

namespace sdm {
int launch_select_f32(const void* kp, const void* qp, const TokenWindow& win, int S, int W, int R,
                      int32_t* idx_w, float* sc_w, int32_t* idx_r, float* sc_r, cudaStream_t s,
                      const uint32_t* stair_g) {
  return launch_select_t<float>(kp, qp, win, S, W, R, idx_w, sc_w, idx_r, sc_r, s, stair_g);
}
}  // namespace sdm
