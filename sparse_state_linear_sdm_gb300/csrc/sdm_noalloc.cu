// Scan entry point for callers that must not allocate device memory.
//
// sdm_scan_forward needs a workspace the caller allocates.  Some callers cannot do that
// at the point where they run the scan: a serving loop or real-time runtime that forbids
// allocation on its request path (an allocation can block, fragment a pre-reserved pool,
// or synchronise the device), or a host application that hands this library a fixed set
// of buffers and owns no allocator at all.  sdm_scan_forward_noalloc serves them with a
// fixed scratch that lives in this library's device image instead.
//
// The scratch is a file-scope __device__ array, so every GPU on which the library is
// loaded keeps SDM_NOALLOC_SCRATCH_BYTES of device memory reserved for it until the
// process exits.  Host code must not use the array's name as a pointer (on the host it
// only stands for the symbol); its device address is looked up once per device with
// cudaGetSymbolAddress, the first time the entry point runs on that device, and cached for
// the life of the process (a cudaDeviceReset reloads the device image, after which the
// cached address is stale: the header tells callers not to use this entry point on that
// device again).
#include <mutex>

#include "sdm_internal.cuh"

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[SDM_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch on the current device (looked up on first use).
int scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SDM_ECUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
      return SDM_ECUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return SDM_OK;
}

}  // namespace

extern "C" int sdm_scan_forward_noalloc(float* M, const int32_t* idx_w, const float* sc_w,
                                        const int32_t* idx_r, const float* sc_r, const void* v,
                                        int v_dt, const float* alpha, const float* beta, int B,
                                        int H, int T, long long N, int d_v, int W, int R,
                                        float* o, int* dev_err, void* stream) {
  // Every check runs on the host before anything is launched: the arguments as
  // sdm_scan_forward checks them, then the record bytes against the fixed scratch.
  int st = sdm::check_scan_args(M, idx_w, sc_w, idx_r, sc_r, v, v_dt, alpha, beta, B, H, T, N,
                                d_v, W, R, o);
  if (st != SDM_OK) return st;
  if (dev_err && (reinterpret_cast<uintptr_t>(dev_err) & 3u)) return SDM_EALIGN;
  size_t need = 0;
  if (T > 0 && !sdm::scan_workspace_bytes(B, H, T, d_v, W, R, &need)) return SDM_EUNSUPPORTED;
  if (need > size_t(SDM_NOALLOC_SCRATCH_BYTES)) return SDM_ESCRATCH;
  void* ws = nullptr;
  if (T > 0) {
    st = scratch_address(&ws);
    if (st != SDM_OK) return st;
  }
  // The planning kernel writes every record field the scan kernel reads, so nothing in
  // the scratch has to start at zero; what the previous call left there is overwritten.
  return sdm_scan_forward(M, idx_w, sc_w, idx_r, sc_r, v, v_dt, alpha, beta, B, H, T, N, d_v, W,
                          R, o, ws, size_t(SDM_NOALLOC_SCRATCH_BYTES), dev_err, stream);
}
