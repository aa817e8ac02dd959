// One decode token for a batch of sequences in a single kernel (Sparse Delta Memory
// technical summary, gist.science/it/paper/2607.07386, "Meccanismo Core" items 2-4, with
// T = 1): product-key selection, the planning of the token, and the gated delta write and
// read of its rows, with the state resident in HBM.
//
// The three-kernel path (sdm_select, planning, scan) spends most of a decode step in
// launch and dependency latency: three small grids, each waiting for the previous one's
// writes.  Here one block per (b, h, 32-column slice of d_v) does all of it:
//   1. the selection of (b, h): warps 0-1 take the k' task, warps 2-3 the q' task (one
//      half each, as the selection kernel's pair mode), written to idx/sc as sdm_select
//      does.  Every slice block of a (b, h) selects the same slots (the work is small and
//      the blocks would otherwise wait for each other).
//   2. the planning of the one token: softmax of the selected write and read scores (the
//      same warp routine as the planning kernel), the source of every row (HBM, or the
//      updated row of the token's own write set for a read slot it also writes), and the
//      device error checks.
//   3. the scan of the token on the block's columns with the scan kernel's thread mapping
//      and arithmetic: gather, forget gate and delta update, write-back, forwarding,
//      weighted read reduced in the same order.  The column width of a block is the one
//      the scan kernel would use for these sizes (choose_scan_shape), so the read's sum
//      runs in the same order too.
// So every output is bit-identical to the three-kernel path.
#include "sdm_select_impl.cuh"

namespace sdm {
namespace {

constexpr int kDecThreads = 256;
constexpr int kDecWarps = kDecThreads / 32;

struct DecodeArgs {
  SelectArgs sel;  // one token per (b, h): items = B * H, Tc = T_total = 1
  const void* v;
  const float* alpha;
  const float* beta;
  float* M;
  float* o;
  long long N;
  int d_v, W, R, slices;
  int cols;  // columns of d_v per block (4 .. 64), as the scan kernel's shape
  size_t sel_smem;  // bytes of the selection's shared memory
  int* dev_err;
};

__host__ __device__ inline size_t decode_scan_smem(int W, int R, int C) {
  const int WR = W + R, WRa = (WR + 3) & ~3;
  return size_t(WR) * C * 4 + size_t(WRa) * 4 /* weights */ + size_t(WRa) * 4 /* slots */ +
         size_t(WRa) * 2 /* sources */ + 16 + size_t(kDecWarps) * C * 4 /* reduction */;
}

template <typename Tv>
__device__ __forceinline__ float v_at(const Tv* p, size_t i);
template <>
__device__ __forceinline__ float v_at<float>(const float* p, size_t i) {
  return p[i];
}
template <>
__device__ __forceinline__ float v_at<uint16_t>(const uint16_t* p, size_t i) {
  return __uint_as_float(uint32_t(p[i]) << 16);
}

__device__ __forceinline__ void cp16(float* dst, const float* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(static_cast<uint32_t>(
                   __cvta_generic_to_shared(dst))),
               "l"(src)
               : "memory");
}

template <typename Tin, typename Tv, int EMAX>
__global__ void __launch_bounds__(kDecThreads, 1) decode_kernel(DecodeArgs d) {
  extern __shared__ __align__(16) unsigned char smem[];
  const SelectArgs& a = d.sel;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int C = d.cols, LPR = C / 4, RPP = kDecThreads / LPR;
  const int bh = blockIdx.x / d.slices;
  const int c0 = (blockIdx.x - bh * d.slices) * C;
  const int W = d.W, R = d.R, WR = W + R, d_v = d.d_v;

  // ---- 1. selection of token (bh, 0) -------------------------------------------------
  {
    const SelectSmem m = select_smem(a, smem);
    select_build_stairs(a, m);
    if (warp < 4) {
      const long long task = 2LL * bh + (warp >> 1);
      select_tasks<Tin, EMAX, true>(a, m, task, task + 1);
    }
  }
  __syncthreads();  // idx / sc of the token written (global, this block)

  // ---- 2. planning of the token (shared memory reused) --------------------------------
  const int WRa = (WR + 3) & ~3;
  float* rows = reinterpret_cast<float*>(smem);        // [WR][C]
  float* wts = rows + size_t(WR) * C;                  // [WRa]
  int32_t* idx = reinterpret_cast<int32_t*>(wts + WRa);  // [WRa]
  int16_t* src = reinterpret_cast<int16_t*>(idx + WRa);  // [WRa]
  float* red = reinterpret_cast<float*>(
      smem + ((size_t(WR) * C * 4 + size_t(WRa) * 10 + 15) / 16 * 16));  // [warps][C]
  const int32_t* gw = a.idx_w + size_t(bh) * W;
  const int32_t* gr = a.idx_r + size_t(bh) * R;
  for (int e = tid; e < WR; e += kDecThreads) idx[e] = e < W ? gw[e] : gr[e - W];
  if (warp == 0) warp_softmax(a.sc_w + size_t(bh) * W, W, wts);
  if (warp == 1) warp_softmax(a.sc_r + size_t(bh) * R, R, wts + W);
  const float alpha = d.alpha[bh], beta = d.beta[bh];
  const int c4 = tid % LPR;
  const Tv* vsrc = static_cast<const Tv*>(d.v) + size_t(bh) * d_v + c0 + 4 * c4;
  const float4 vv = make_float4(v_at<Tv>(vsrc, 0), v_at<Tv>(vsrc, 1), v_at<Tv>(vsrc, 2),
                                v_at<Tv>(vsrc, 3));
  __syncthreads();
  int errs = 0;
  for (int e = tid; e < WR; e += kDecThreads) {
    const int32_t x = idx[e];
    int code = -1;
    if (x < 0 || x >= d.N) {
      code = -2;
      errs |= SDM_DEV_INDEX_RANGE;
    } else if (e < W) {
      for (int p = 0; p < W; ++p)
        if (p != e && idx[p] == x) errs |= SDM_DEV_DUP_WRITE;
    } else {
      for (int p = 0; p < W; ++p)  // a read of a row this token writes: the updated row
        if (idx[p] == x) {
          code = p;
          break;
        }
    }
    src[e] = int16_t(code);
  }
  if (errs && d.dev_err) atomicOr(d.dev_err, errs);
  __syncthreads();

  // ---- 3. the token's scan on columns c0 .. c0+C-1 -------------------------------------
  float* Mbh = d.M + size_t(bh) * size_t(d.N) * d_v + c0;
  for (int e = tid / LPR; e < WR; e += RPP)
    if (src[e] == -1) cp16(rows + e * C + 4 * c4, Mbh + size_t(idx[e]) * d_v + 4 * c4);
  asm volatile("cp.async.commit_group;\ncp.async.wait_group 0;" ::: "memory");
  __syncthreads();

  // Forget gate and delta update of the W write rows (in shared memory and in HBM).
  for (int e = tid / LPR; e < W; e += RPP) {
    if (src[e] == -2) continue;
    float4* cell = reinterpret_cast<float4*>(rows + e * C) + c4;
    const float4 m = *cell;
    const float kb = beta * wts[e];
    float4 r;
    float mt_;
    mt_ = alpha * m.x; r.x = fmaf(kb, vv.x - mt_, mt_);
    mt_ = alpha * m.y; r.y = fmaf(kb, vv.y - mt_, mt_);
    mt_ = alpha * m.z; r.z = fmaf(kb, vv.z - mt_, mt_);
    mt_ = alpha * m.w; r.w = fmaf(kb, vv.w - mt_, mt_);
    *cell = r;
    *(reinterpret_cast<float4*>(Mbh + size_t(idx[e]) * d_v) + c4) = r;
  }
  __syncthreads();

  // Read rows this token also writes take the updated row.
  for (int e = W + tid; e < WR; e += kDecThreads) {
    const int code = src[e];
    if (code >= 0 && code < W) {
      const float4* from = reinterpret_cast<const float4*>(rows + code * C);
      float4* to = reinterpret_cast<float4*>(rows + e * C);
      for (int q = 0; q < LPR; ++q) to[q] = from[q];
    }
  }
  __syncthreads();

  // Weighted read of the R read rows (after the write), reduced in the scan kernel's order.
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int e = tid / LPR; e < R; e += RPP) {
    if (src[W + e] == -2) continue;
    const float r = wts[W + e];
    const float4 m = reinterpret_cast<const float4*>(rows + (W + e) * C)[c4];
    acc.x = fmaf(r, m.x, acc.x);
    acc.y = fmaf(r, m.y, acc.y);
    acc.z = fmaf(r, m.z, acc.z);
    acc.w = fmaf(r, m.w, acc.w);
  }
  for (int off = LPR; off < 32; off <<= 1) {
    acc.x += __shfl_xor_sync(0xFFFFFFFFu, acc.x, off);
    acc.y += __shfl_xor_sync(0xFFFFFFFFu, acc.y, off);
    acc.z += __shfl_xor_sync(0xFFFFFFFFu, acc.z, off);
    acc.w += __shfl_xor_sync(0xFFFFFFFFu, acc.w, off);
  }
  if (lane < LPR) reinterpret_cast<float4*>(red + warp * C)[lane] = acc;
  __syncthreads();
  if (tid < LPR) {
    float4 s = reinterpret_cast<const float4*>(red)[tid];
#pragma unroll
    for (int w = 1; w < kDecWarps; ++w) {
      const float4 t = reinterpret_cast<const float4*>(red + w * C)[tid];
      s = make_float4(s.x + t.x, s.y + t.y, s.z + t.z, s.w + t.w);
    }
    *(reinterpret_cast<float4*>(d.o + size_t(bh) * d_v + c0) + tid) = s;
  }
}

// Launch shape of the decode kernel: column width (the scan kernel's), blocks, shared memory.
template <typename Tin>
int decode_shape(int BH, int S, int d_v, int W, int R, SelectArgs* sel, int* cols, size_t* smem,
                 size_t* sel_smem) {
  ScanShape shape;
  const int st = choose_scan_shape(BH, d_v, W, R, 0, 0, &shape);
  if (st != SDM_OK) return st;
  if (shape.cols < 4 || shape.cols > 64 || d_v % shape.cols != 0) return SDM_EUNSUPPORTED;
  size_t stair_bytes = 0, per_warp = 0;
  select_args<Tin>(nullptr, nullptr, whole_sequences(BH, 1), S, W, R, nullptr, nullptr, nullptr,
                   nullptr, sel, &stair_bytes, &per_warp);
  sel->warps = 4;
  *cols = shape.cols;
  *sel_smem = stair_bytes + 4 * per_warp;
  *smem = *sel_smem;
  const size_t scan_smem = decode_scan_smem(W, R, shape.cols);
  if (scan_smem > *smem) *smem = scan_smem;
  int dev = 0, max_smem = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
    return SDM_ECUDA;
  return *smem > size_t(max_smem) ? SDM_EUNSUPPORTED : SDM_OK;
}

template <typename Tin>
int launch_decode_t(const void* kp, const void* qp, const void* v, int v_dt, const float* alpha,
                    const float* beta, float* M, int BH, int S, int d_v, int W, int R,
                    int32_t* idx_w, float* sc_w, int32_t* idx_r, float* sc_r, float* o,
                    int* dev_err, cudaStream_t s) {
  DecodeArgs dargs;
  int cols = 0;
  size_t smem = 0;
  const int st = decode_shape<Tin>(BH, S, d_v, W, R, &dargs.sel, &cols, &smem, &dargs.sel_smem);
  if (st != SDM_OK) return st;
  dargs.sel.kp = kp;
  dargs.sel.qp = qp;
  dargs.sel.idx_w = idx_w;
  dargs.sel.sc_w = sc_w;
  dargs.sel.idx_r = idx_r;
  dargs.sel.sc_r = sc_r;
  dargs.v = v;
  dargs.alpha = alpha;
  dargs.beta = beta;
  dargs.M = M;
  dargs.o = o;
  dargs.N = (long long)S * S;
  dargs.d_v = d_v;
  dargs.W = W;
  dargs.R = R;
  dargs.cols = cols;
  dargs.slices = d_v / cols;
  dargs.dev_err = dev_err;
  const bool big = W > 128 || R > 128;
  const void* fn;
  if (v_dt == SDM_BF16)
    fn = big ? reinterpret_cast<const void*>(&decode_kernel<Tin, uint16_t, 32>)
             : reinterpret_cast<const void*>(&decode_kernel<Tin, uint16_t, 4>);
  else
    fn = big ? reinterpret_cast<const void*>(&decode_kernel<Tin, float, 32>)
             : reinterpret_cast<const void*>(&decode_kernel<Tin, float, 4>);
  if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)) !=
      cudaSuccess)
    return SDM_ECUDA;
  const long long blocks = (long long)BH * dargs.slices;
  if (blocks > 0x7FFFFFFFLL) return SDM_EUNSUPPORTED;
  void* args[] = {&dargs};
  if (cudaLaunchKernel(fn, dim3(unsigned(blocks)), dim3(kDecThreads), args, smem, s) != cudaSuccess)
    return SDM_ECUDA;
  return last_launch_status();
}

}  // namespace

int launch_decode(const void* kp, const void* qp, int in_dt, const void* v, int v_dt,
                  const float* alpha, const float* beta, float* M, int BH, int S, int d_v, int W,
                  int R, int32_t* idx_w, float* sc_w, int32_t* idx_r, float* sc_r, float* o,
                  int* dev_err, cudaStream_t s) {
  if (BH == 0) return SDM_OK;
  return in_dt == SDM_BF16
             ? launch_decode_t<uint16_t>(kp, qp, v, v_dt, alpha, beta, M, BH, S, d_v, W, R, idx_w,
                                         sc_w, idx_r, sc_r, o, dev_err, s)
             : launch_decode_t<float>(kp, qp, v, v_dt, alpha, beta, M, BH, S, d_v, W, R, idx_w,
                                      sc_w, idx_r, sc_r, o, dev_err, s);
}

int decode_supported(int in_dt, int BH, int S, int d_v, int W, int R) {
  SelectArgs sel;
  int cols = 0;
  size_t smem = 0, sel_smem = 0;
  return in_dt == SDM_BF16 ? decode_shape<uint16_t>(BH, S, d_v, W, R, &sel, &cols, &smem, &sel_smem)
                           : decode_shape<float>(BH, S, d_v, W, R, &sel, &cols, &smem, &sel_smem);
}

}  // namespace sdm
