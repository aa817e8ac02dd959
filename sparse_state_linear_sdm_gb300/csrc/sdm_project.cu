// Projection of the token features onto the product-key halves, on the tcgen05 tensor
// cores (Sparse Delta Memory technical summary, gist.science/it/paper/2607.07386,
// "Meccanismo Core" item 2: the projected key k' and query q' whose halves are the
// sub-scores; "Design IsoFLOP": the projections are plain linear layers).
//
//   k'[b,h,t,half,s] = sum_d x[b,t,d] w[(h*2 + half)*S + s, d]
//   q'[b,h,t,half,s] = sum_d x[b,t,d] w[H*2*S + (h*2 + half)*S + s, d]
//
// is one GEMM  Y[m, n] = sum_d X[m, d] W[n, d]  over the m = b*T + t token rows and the
// n < 2*H*2S output columns: bf16 operands, fp32 accumulation, rounded to bf16 (nearest
// even) and stored straight into the [B,H,T,2,S] layout the selection reads, so no
// transpose pass follows.
//
// Kernels: persistent, one CTA per SM, K in steps of 64 (one 128-byte swizzle atom of bf16),
// two launch shapes of the same warp roles:
//   warp 0      TMA producer: X and W tiles, 128-byte swizzled, into a ring of stages in
//               shared memory
//   warp 1      TMEM owner (512 columns: two 256-column fp32 accumulators) and MMA issuer
//               (one thread); tcgen05.commit frees a stage and, after a tile's last stage,
//               hands the accumulator to the epilogue
//   warps 2..5  epilogue: each warp reads its 32 TMEM lanes (= 32 rows of the tile) with
//               tcgen05.ld, converts to bf16 and stores 16-byte pieces of the row, while the
//               other accumulator is filled by the next tile's MMAs
// (0) single CTAs: 128 x 256 tiles, tcgen05.mma M128 N256, 4 stages of 48 KB;
// (2) the default: CTA pairs whose MMAs form one 256 x 256 tile (tcgen05.mma cta_group::2
//     M256 N256, issued by the even CTA), each CTA staging only its 128 rows of X and half
//     of the W tile (6 stages of 32 KB), which halves the operand bytes each SM's shared
//     memory takes in and hands to the tensor core per flop.
// All 256 columns of a tile lie in one head's k' or q' when S % 128 == 0.  Tiles run in
// groups of row tiles (see unit_coords), so the CTAs running at once share rows of X and
// column tiles of W in L2.
// Every mbarrier wait is bounded in time: an expired wait raises a CTA-wide stop flag,
// every role leaves its loop, outstanding copies and MMAs are waited for (bounded), TMEM
// is freed and SDM_DEV_TIMEOUT is reported through dev_err.
#include "sdm_internal.cuh"
#include "sdm_select_count.cuh"

#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include <mutex>

namespace sdm {
namespace {

constexpr int BM = 128, BN = 256, BK = 64, STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;  // 16 KB
constexpr int B_BYTES = BN * BK * 2;  // 32 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int kThreads = 192;
constexpr uint32_t kTmemCols = 2 * BN;
constexpr int kNumBars = 2 * STAGES + 5;  // full[], empty[], acc_full[2], acc_empty[2], drain
constexpr int kSmemBytes = STAGES * STAGE_BYTES + 1024 /* alignment slack */ + 256;
constexpr unsigned long long kWaitNs = 2000000000ull;  // 2 s per wait
constexpr int kGroup = 32;  // row-tile pairs per group of the tile order (measured best of 1..64)

// Instruction descriptor of tcgen05.mma kind::f16: D fp32 (bits 4-5 = 1), A and B bf16
// (bits 7-9 = 1, 10-12 = 1), both K-major (bits 15, 16 = 0), N >> 3 at bits 17-22,
// M >> 4 at bits 24-28.
constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | (uint32_t(BN >> 3) << 17) |
                            (uint32_t(BM >> 4) << 24);

struct ProjArgs {
  int Mrows, Ncols, D;
  int T, H, S;
  uint16_t* kp;
  uint16_t* qp;
  int* dev_err;
  unsigned long long wait_ns;  // time limit of every wait (kWaitNs outside tests)
  int stall_cta;               // tests only: this cluster rank's producer stops issuing after
  int stall_step;              // stall_step K steps (-1: never), so that a wait runs out
};

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
// Counts `bytes` of the current phase's transactions as done without a copy.
__device__ __forceinline__ void mbar_complete_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.complete_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Waits until the barrier's phase of the given parity has completed.  Returns false when
// the CTA's stop flag is up or the wait ran past its time limit (then it raises the flag).
__device__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* stop,
                          unsigned long long limit_ns = kWaitNs) {
  if (mbar_test(bar, parity)) return true;
  const unsigned long long t0 = global_ns();
  for (uint32_t i = 1; i < (1u << 28); ++i) {
    if (mbar_test(bar, parity)) return true;
    if ((i & 31u) == 0) {
      if (*stop) return false;
      if (global_ns() - t0 > limit_ns) break;
    }
  }
  *stop = 1;
  return false;
}

// One bounded wait of mbar_wait on a barrier of its own, for checking the timeout path
// without a kernel that can hang: mode 0 waits on a phase that nothing completes (the wait
// runs out after limit_ns), mode 1 on a phase its own arrival has completed, mode 2 with
// the stop flag already raised (as when another role of the CTA gave up first).  Like the
// projection kernel, it reports SDM_DEV_TIMEOUT through dev_err when the stop flag is up at
// the end.  One warp; no copies or MMAs are issued, so nothing is in flight at exit.
__global__ void bounded_wait_kernel(int mode, unsigned long long limit_ns, int* dev_err,
                                    unsigned long long* elapsed_ns) {
  __shared__ __align__(8) uint64_t bar_mem;
  __shared__ int stop;
  if (threadIdx.x != 0) return;
  const uint32_t bar = smem_u32(&bar_mem);
  stop = mode == 2 ? 1 : 0;
  mbar_init(bar, 1);  // initialised, arrived on and waited on by this one thread
  if (mode == 1) mbar_arrive(bar);
  const unsigned long long t0 = global_ns();
  mbar_wait(bar, 0, &stop, limit_ns);
  if (elapsed_ns) *elapsed_ns = global_ns() - t0;
  if (stop && dev_err) atomicOr(dev_err, SDM_DEV_TIMEOUT);
}

// Teardown wait: only the time limit, not the stop flag.
__device__ void mbar_wait_teardown(uint32_t bar, uint32_t parity) {
  const unsigned long long t0 = global_ns();
  for (uint32_t i = 0; i < (1u << 28); ++i) {
    if (mbar_test(bar, parity)) return;
    if ((i & 31u) == 31u && global_ns() - t0 > kWaitNs) return;
  }
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

// Shared-memory matrix descriptor of a K-major operand tile in the 128-byte swizzle layout
// written by TMA: rows of 128 bytes, 8-row atoms of 1,024 bytes stacked along M/N (stride
// byte offset 1,024; the leading byte offset is not used by this layout), descriptor
// version 1 at bit 46, swizzle mode 2 (128 bytes) at bits 61-63.  The K step of 16
// elements inside the atom advances the start address by 32 bytes.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  return uint64_t((saddr & 0x3FFFFu) >> 4) | (uint64_t(1) << 16) | (uint64_t(1024 >> 4) << 32) |
         (uint64_t(1) << 46) | (uint64_t(2) << 61);
}

__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %3, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %4, p;\n}\n" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(accumulate), "r"(kIdesc)
      : "memory");
}
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// 32 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_load32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32"
      " {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15,"
      " %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31},"
      " [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ uint32_t pack_bf16(uint32_t lo, uint32_t hi) {
  const __nv_bfloat162 p = __floats2bfloat162_rn(__uint_as_float(lo), __uint_as_float(hi));
  return *reinterpret_cast<const uint32_t*>(&p);
}

// Stores columns n .. n+31 of token row (b, t).  VEC: 2S % 8 == 0 and 16-byte aligned
// outputs, so every 8-column piece lies in one (k' or q', head) block and is one 16-byte
// store; otherwise column by column.
template <bool VEC>
__device__ __forceinline__ void store_cols(const ProjArgs& a, int b, int t, int n,
                                           const uint32_t (&r)[32]) {
  const int S2 = 2 * a.S, HS2 = a.H * S2;
  if (VEC) {
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      const int c = n + 8 * g;
      if (c >= a.Ncols) break;
      const int which = c >= HS2;
      const int rem = c - which * HS2;
      const int h = rem / S2, cc = rem - h * S2;
      uint16_t* dst = (which ? a.qp : a.kp) + ((size_t(b) * a.H + h) * a.T + t) * S2 + cc;
      uint4 v;
      v.x = pack_bf16(r[8 * g + 0], r[8 * g + 1]);
      v.y = pack_bf16(r[8 * g + 2], r[8 * g + 3]);
      v.z = pack_bf16(r[8 * g + 4], r[8 * g + 5]);
      v.w = pack_bf16(r[8 * g + 6], r[8 * g + 7]);
      *reinterpret_cast<uint4*>(dst) = v;
    }
  } else {
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      const int c = n + j;
      if (c >= a.Ncols) continue;
      const int which = c >= HS2;
      const int rem = c - which * HS2;
      const int h = rem / S2, cc = rem - h * S2;
      uint16_t* dst = (which ? a.qp : a.kp) + ((size_t(b) * a.H + h) * a.T + t) * S2 + cc;
      const __nv_bfloat16 v = __float2bfloat16_rn(__uint_as_float(r[j]));
      *dst = *reinterpret_cast<const uint16_t*>(&v);
    }
  }
}

// Work unit u -> (row-tile pair mp, column tile n): groups of kGroup row-tile pairs, the
// pairs of a group fastest, then the column tiles, so that the units running at the same
// time share a few rows of X and a few column tiles of W in L2.
__device__ __forceinline__ void unit_coords(int u, int MP, int NT, int& mp, int& n) {
  const int per_group = kGroup * NT;
  const int g = u / per_group, w = u - g * per_group;
  const int gm = min(kGroup, MP - g * kGroup);
  n = w / gm;
  mp = g * kGroup + (w - n * gm);
}

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release;\nbarrier.cluster.wait.acquire;" ::: "memory");
}

// Single CTAs: each loads its X rows and its whole W tile per stage; work units are
// (row tile, column tile) pairs.
template <bool VEC>
__global__ void __launch_bounds__(kThreads, 1)
    project_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                   ProjArgs a) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t ring = (raw + 1023u) & ~1023u;  // stage tiles on 1,024-byte swizzle atoms
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem_raw + (ring - raw) + STAGES * STAGE_BYTES);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + kNumBars);
  volatile int* stop = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const int FULL = 0, EMPTY = STAGES, ACC_FULL = 2 * STAGES, ACC_EMPTY = 2 * STAGES + 2,
            DRAIN = 2 * STAGES + 4;
  auto bar = [&](int i) { return smem_u32(bars + i); };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int cid = blockIdx.x, ncl = gridDim.x;
  const int NT = (a.Ncols + BN - 1) / BN;
  const int MP = (a.Mrows + BM - 1) / BM;
  const int units = MP * NT;
  const int KB = (a.D + BK - 1) / BK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(bar(FULL + s), 1);
      mbar_init(bar(EMPTY + s), 1);  // the MMA thread's commit
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(ACC_FULL + i), 1);
      mbar_init(bar(ACC_EMPTY + i), 4);  // one arrival per epilogue warp
    }
    mbar_init(bar(DRAIN), 1);
    *stop = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmX)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmW)) : "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_slot)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  uint32_t used = 0, last_par = 0;  // producer: per stage, ever loaded / parity of its last load
  if (warp == 0) {
    if (lane == 0) {
      // ---- TMA producer ----
      int stage = 0, issued = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int u = cid; ok && u < units; u += ncl) {
        int mp, n;
        unit_coords(u, MP, NT, mp, n);
        const int m0 = mp * BM, n0 = n * BN;
        for (int kb = 0; kb < KB; ++kb) {
          if (a.stall_cta == 0 && issued >= a.stall_step) {
            ok = false;
            break;
          }
          if (!mbar_wait(bar(EMPTY + stage), phase ^ 1u, stop, a.wait_ns)) {
            ok = false;
            break;
          }
          ++issued;
          const uint32_t sa = ring + uint32_t(stage) * STAGE_BYTES;
          mbar_expect_tx(bar(FULL + stage), STAGE_BYTES);
          tma_load_2d(sa, &tmX, kb * BK, m0, bar(FULL + stage));
          tma_load_2d(sa + A_BYTES, &tmW, kb * BK, n0, bar(FULL + stage));
          tma_load_2d(sa + A_BYTES + B_BYTES / 2, &tmW, kb * BK, n0 + BN / 2, bar(FULL + stage));
          used |= 1u << stage;
          last_par = (last_par & ~(1u << stage)) | (phase << stage);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---- MMA issuer ----
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      int it = 0;
      for (int u = cid; ok && u < units; u += ncl, ++it) {
        const int acc = it & 1;
        const uint32_t acc_par = uint32_t(it >> 1) & 1u;
        if (!mbar_wait(bar(ACC_EMPTY + acc), acc_par ^ 1u, stop, a.wait_ns)) break;
        tc_fence_after();
        const uint32_t d = tmem_base + uint32_t(acc * BN);
        for (int kb = 0; kb < KB; ++kb) {
          if (!mbar_wait(bar(FULL + stage), phase, stop, a.wait_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = ring + uint32_t(stage) * STAGE_BYTES;
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk)
            mma_bf16(d, sw128_desc(sa + kk * 32), sw128_desc(sa + A_BYTES + kk * 32),
                     (kb | kk) != 0);
          mma_commit(bar(EMPTY + stage));
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (ok) mma_commit(bar(ACC_FULL + acc));
      }
      // Every MMA issued has finished before TMEM and shared memory are released.
      mma_commit(bar(DRAIN));
      mbar_wait_teardown(bar(DRAIN), 0);
    }
  } else {
    // ---- epilogue: warp w reads TMEM lanes 32*(w % 4) .. +31 ----
    const int quad = warp & 3;
    const int row = quad * 32 + lane;
    int it = 0;
    for (int u = cid; u < units; u += ncl, ++it) {
      const int acc = it & 1;
      const uint32_t acc_par = uint32_t(it >> 1) & 1u;
      // every lane waits; the warp leaves together (tcgen05.ld needs the whole warp)
      if (!__all_sync(0xFFFFFFFFu, mbar_wait(bar(ACC_FULL + acc), acc_par, stop, a.wait_ns))) break;
      tc_fence_after();
      int mp, n;
      unit_coords(u, MP, NT, mp, n);
      const int m = mp * BM + row, n0 = n * BN;
      const int b = m / a.T, t = m - b * a.T;
      const uint32_t taddr = tmem_base + (uint32_t(quad * 32) << 16) + uint32_t(acc * BN);
#pragma unroll 1
      for (int c = 0; c < BN / 32; ++c) {
        uint32_t r[32];
        tmem_load32(taddr + uint32_t(c * 32), r);
        if (m < a.Mrows && n0 + c * 32 < a.Ncols) store_cols<VEC>(a, b, t, n0 + c * 32, r);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(ACC_EMPTY + acc));
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                 "r"(kTmemCols)
                 : "memory");
  // After a stop, whichever role raised it, every copy issued lands before the CTA's shared
  // memory goes away: the last phase of each stage the producer loaded has completed.
  if (warp == 0 && lane == 0 && *stop)
    for (int s = 0; s < STAGES; ++s)
      if (used & (1u << s)) mbar_wait_teardown(bar(FULL + s), (last_par >> s) & 1u);
  if (threadIdx.x == 0 && *stop && a.dev_err) atomicOr(a.dev_err, SDM_DEV_TIMEOUT);
}

// ---- 2-SM variant: one tcgen05.mma.cta_group::2 M256 x N256 per K16 for a CTA pair ----
//
// The even CTA of a cluster of two (the leader) issues the MMAs for both: A rows 0-127 come
// from its own shared memory and rows 128-255 from its peer's (same offset), the W tile's
// rows 0-127 from the leader and 128-255 from the peer, and each CTA's TMEM receives its own
// 128 rows of the 256 x 256 accumulator.  Each CTA stages only its own X rows and its half of
// the W tile (32 KB per stage, 6 stages).  Both CTAs' copies complete on the leader's full
// barrier; the leader's commits arrive on the empty and accumulator-full barriers of both
// CTAs; the epilogue warps of both arrive on the leader's accumulator-empty barrier.
constexpr int STAGES2 = 6;
constexpr int STAGE2_BYTES = A_BYTES + B_BYTES / 2;
constexpr int kSmemBytes2 = STAGES2 * STAGE2_BYTES + 1024 + 256;  // + barriers, flags, counts
constexpr int kNumBars2 = 2 * STAGES2 + 5;
constexpr uint32_t kIdesc2 = (1u << 4) | (1u << 7) | (1u << 10) | (uint32_t(BN >> 3) << 17) |
                             (uint32_t((2 * BM) >> 4) << 24);

__device__ __forceinline__ uint32_t cluster_addr(uint32_t local, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
  return r;
}
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_bar) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_bar)
               : "memory");
}
__device__ __forceinline__ bool mbar_test_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ uint32_t ld_cluster_u32(uint32_t cluster_addr) {
  uint32_t v;
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(cluster_addr) : "memory");
  return v;
}
__device__ __forceinline__ void st_cluster_u32(uint32_t cluster_addr, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(cluster_addr), "r"(v) : "memory");
}
// mbar_wait with cluster-scope acquire (barriers that the peer CTA arrives on).  Giving up
// raises the stop flags of both CTAs of the pair (peer_stop: the peer's flag).
__device__ bool mbar_wait_cluster(uint32_t bar, uint32_t parity, volatile int* stop,
                                  uint32_t peer_stop, unsigned long long limit_ns) {
  if (mbar_test_cluster(bar, parity)) return true;
  const unsigned long long t0 = global_ns();
  for (uint32_t i = 1; i < (1u << 28); ++i) {
    if (mbar_test_cluster(bar, parity)) return true;
    if ((i & 31u) == 0) {
      if (*stop) return false;
      if (global_ns() - t0 > limit_ns) break;
    }
  }
  *stop = 1;
  st_cluster_u32(peer_stop, 1u);
  return false;
}
// A box loaded into this CTA's shared memory, completing on a barrier of either CTA of the pair.
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* map, int x, int y,
                                                 uint32_t cluster_bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".cta_group::2 [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(cluster_bar)
      : "memory");
}
__device__ __forceinline__ void mma2_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %3, 0;\n"
      " tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %4, p;\n}\n" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(accumulate), "r"(kIdesc2)
      : "memory");
}
__device__ __forceinline__ void mma2_commit_both(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(bar),
      "h"(uint16_t(0x3))
      : "memory");
}
__device__ __forceinline__ void mma2_commit_local(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   bar)
               : "memory");
}

template <bool VEC>
__global__ void __launch_bounds__(kThreads, 1)
    project_kernel_2sm(const __grid_constant__ CUtensorMap tmX,
                       const __grid_constant__ CUtensorMap tmW, ProjArgs a) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t ring = (raw + 1023u) & ~1023u;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem_raw + (ring - raw) + STAGES2 * STAGE2_BYTES);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + kNumBars2);
  volatile int* stop = reinterpret_cast<volatile int*>(tmem_slot + 1);
  // Copies this CTA's producer issued per stage (read by the leader after a stop).
  volatile uint32_t* issued = tmem_slot + 2;
  const int FULL = 0, EMPTY = STAGES2, ACC_FULL = 2 * STAGES2, ACC_EMPTY = 2 * STAGES2 + 2,
            DRAIN = 2 * STAGES2 + 4;
  auto bar = [&](int i) { return smem_u32(bars + i); };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  const bool leader = rank == 0;
  const uint32_t peer_stop = cluster_addr(smem_u32(const_cast<int*>(stop)), rank ^ 1u);
  const int cid = blockIdx.x / 2, ncl = gridDim.x / 2;
  const int NT = (a.Ncols + BN - 1) / BN;
  const int MP = ((a.Mrows + BM - 1) / BM + 1) / 2;
  const int units = MP * NT;
  const int KB = (a.D + BK - 1) / BK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES2; ++s) {
      mbar_init(bar(FULL + s), 1);   // the leader's expect_tx; both CTAs' bytes
      mbar_init(bar(EMPTY + s), 1);  // the leader's commit
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(ACC_FULL + i), 1);
      mbar_init(bar(ACC_EMPTY + i), 8);  // the 4 epilogue warps of each CTA
    }
    mbar_init(bar(DRAIN), 1);
    *stop = 0;
    for (int s = 0; s < STAGES2; ++s) issued[s] = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmX)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmW)) : "memory");
  }
  if (warp == 1) {  // one warp of each CTA of the pair allocates, together
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_slot)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      // ---- TMA producer (both CTAs) ----
      int stage = 0, steps = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int u = cid; ok && u < units; u += ncl) {
        int mp, n;
        unit_coords(u, MP, NT, mp, n);
        const int m0 = (mp * 2 + int(rank)) * BM, n0 = n * BN;
        for (int kb = 0; kb < KB; ++kb) {
          if (int(rank) == a.stall_cta && steps >= a.stall_step) {
            ok = false;
            break;
          }
          if (!mbar_wait_cluster(bar(EMPTY + stage), phase ^ 1u, stop, peer_stop, a.wait_ns)) {
            ok = false;
            break;
          }
          ++steps;
          const uint32_t sa = ring + uint32_t(stage) * STAGE2_BYTES;
          const uint32_t full_leader = cluster_addr(bar(FULL + stage), 0);
          if (leader) mbar_expect_tx(bar(FULL + stage), 2 * STAGE2_BYTES);
          tma_load_2d_pair(sa, &tmX, kb * BK, m0, full_leader);
          tma_load_2d_pair(sa + A_BYTES, &tmW, kb * BK, n0 + int(rank) * (BN / 2), full_leader);
          issued[stage] = issued[stage] + 1u;
          if (++stage == STAGES2) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && leader) {
      // ---- MMA issuer (leader only) ----
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      int it = 0;
      for (int u = cid; ok && u < units; u += ncl, ++it) {
        const int acc = it & 1;
        const uint32_t acc_par = uint32_t(it >> 1) & 1u;
        if (!mbar_wait_cluster(bar(ACC_EMPTY + acc), acc_par ^ 1u, stop, peer_stop, a.wait_ns)) break;
        tc_fence_after();
        const uint32_t d = tmem_base + uint32_t(acc * BN);
        for (int kb = 0; kb < KB; ++kb) {
          if (!mbar_wait_cluster(bar(FULL + stage), phase, stop, peer_stop, a.wait_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = ring + uint32_t(stage) * STAGE2_BYTES;
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk)
            mma2_bf16(d, sw128_desc(sa + kk * 32), sw128_desc(sa + A_BYTES + kk * 32),
                      (kb | kk) != 0);
          mma2_commit_both(bar(EMPTY + stage));
          if (++stage == STAGES2) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (ok) mma2_commit_both(bar(ACC_FULL + acc));
      }
      mma2_commit_local(bar(DRAIN));
      mbar_wait_teardown(bar(DRAIN), 0);
    }
  } else {
    // ---- epilogue (both CTAs): warp w reads TMEM lanes 32*(w % 4) .. +31 ----
    const int quad = warp & 3;
    const int row = quad * 32 + lane;
    int it = 0;
    for (int u = cid; u < units; u += ncl, ++it) {
      const int acc = it & 1;
      const uint32_t acc_par = uint32_t(it >> 1) & 1u;
      if (!__all_sync(0xFFFFFFFFu,
                      mbar_wait_cluster(bar(ACC_FULL + acc), acc_par, stop, peer_stop, a.wait_ns)))
        break;
      tc_fence_after();
      int mp, n;
      unit_coords(u, MP, NT, mp, n);
      const int m = (mp * 2 + int(rank)) * BM + row, n0 = n * BN;
      const int b = m / a.T, t = m - b * a.T;
      const uint32_t taddr = tmem_base + (uint32_t(quad * 32) << 16) + uint32_t(acc * BN);
#pragma unroll 1
      for (int c = 0; c < BN / 32; ++c) {
        uint32_t r[32];
        tmem_load32(taddr + uint32_t(c * 32), r);
        if (m < a.Mrows && n0 + c * 32 < a.Ncols) store_cols<VEC>(a, b, t, n0 + c * 32, r);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(cluster_addr(bar(ACC_EMPTY + acc), 0));
    }
  }

  tc_fence_before();
  __syncthreads();
  // Every role of both CTAs has finished: the leader's MMAs into both CTAs' TMEM are done
  // before either frees it, and both producers' copy counts and stop flags are final.
  cluster_sync_all();
  tc_fence_after();
  if (warp == 1)
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                 "r"(kTmemCols)
                 : "memory");
  if (leader && warp == 0 && lane == 0 && *stop) {
    // After a stop, every copy either CTA issued lands before the pair's shared memory goes
    // away.  All copies of a stage complete on the leader's full barrier, which the leader
    // arms with both CTAs' bytes; per stage the two producers issued the same number of
    // copies or one more than the other (each is at most one round of stages ahead of the
    // MMAs, which need both halves).  The leader arms a phase only the peer issued with the
    // peer's bytes, counts the peer's missing bytes of a phase only it issued as done, and
    // waits for the last phase of each stage.
    const uint32_t peer_issued = cluster_addr(smem_u32(const_cast<uint32_t*>(issued)), 1u);
    for (int s = 0; s < STAGES2; ++s) {
      const uint32_t lc = issued[s], pc = ld_cluster_u32(peer_issued + 4u * uint32_t(s));
      if (pc == lc + 1u) {
        mbar_expect_tx(bar(FULL + s), STAGE2_BYTES);
        mbar_wait_teardown(bar(FULL + s), lc & 1u);
      } else if (lc == pc + 1u) {
        mbar_complete_tx(bar(FULL + s), STAGE2_BYTES);
        mbar_wait_teardown(bar(FULL + s), (lc - 1u) & 1u);
      } else if (lc == pc && lc > 0u) {
        mbar_wait_teardown(bar(FULL + s), (lc - 1u) & 1u);
      }
    }
  }
  if (threadIdx.x == 0 && *stop && a.dev_err) atomicOr(a.dev_err, SDM_DEV_TIMEOUT);
  cluster_sync_all();  // the peer's shared memory outlives the leader's drain
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// Row-major bf16 matrix [rows, cols] read in boxes of box_rows x 64 columns, 128-byte swizzle,
// zero fill outside the matrix.
bool bf16_tile_map(CUtensorMap* map, const void* base, int rows, int cols, int box_rows) {
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  const cuuint64_t dims[2] = {cuuint64_t(cols), cuuint64_t(rows)};
  const cuuint64_t strides[1] = {cuuint64_t(cols) * 2};
  const cuuint32_t box[2] = {cuuint32_t(BK), cuuint32_t(box_rows)};
  const cuuint32_t estr[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
  return n;
}


// ---- projection fused with the inner top-k of every half ----------------------------------
//
// "Meccanismo Core" item 2 of the same summary takes the top-k of each half of k' and q';
// here they are taken on chip, straight from the projection's accumulators, so k' and q'
// never reach HBM: only each half's top-kin list (kin = min(W or R, S) packed entries,
// bf16 value << 16 | index) is written, and the outer top-K over the lists' staircase runs
// in a second kernel (outer_kernel below).
//
// Transposed tiles: a work unit is (a block of FT = 64 tokens, one half g), g = (which * H +
// h) * 2 + half, whose S sub-scores are rows [g*S, g*S + S) of W.  The unit's S x 64 outputs
// (sub-scores x tokens) accumulate in TMEM, M-tile mt (128 sub-scores, the MMA's M) in
// columns [64 mt, 64 mt + 64) (S = 1024 fills all 512 columns), so a token's whole half is on
// chip when the K loop ends.  Per K step of 64 the X tile (64 tokens x 64, the MMA's B) is
// loaded once and used by the S/128 MMAs (M128 N64 K16 x 4) of the step; the W tiles stream
// through their own ring.  The epilogue warps then read the accumulators in groups of FG = 8
// tokens, round them to bf16 (nearest even, as the unfused kernel stores them) into a
// staging buffer [8][S] in shared memory, and select each token's top-kin there with the
// counting selection (inner_count_smem; the general path on its rare fallback), two tokens
// per warp.  The accumulation order of every output is the unfused kernel's (K blocks in
// sequence, the same MMA K steps), so the lists are those of sdm_select on sdm_project_kq's
// output.  The MMAs of the next unit wait until the epilogue has read the accumulators.
constexpr int FT = 64;                    // tokens per unit (the MMA's N)
constexpr int FG = 8;                     // tokens per epilogue group
constexpr int F_A_BYTES = 128 * BK * 2;   // 16 KB: W tile (128 sub-scores x 64)
constexpr int F_B_BYTES = FT * BK * 2;    // 8 KB: X tile (64 tokens x 64)
constexpr int F_ASTAGES = 6, F_BSTAGES = 3;
constexpr int F_EPI_WARPS = 4;
constexpr uint32_t kIdescF = (1u << 4) | (1u << 7) | (1u << 10) | (uint32_t(FT >> 3) << 17) |
                             (uint32_t(128 >> 4) << 24);
// barriers: a_full, a_empty, b_full, b_empty, acc_full, tmem_empty, drain
constexpr int F_NUM_BARS = 2 * F_ASTAGES + 2 * F_BSTAGES + 3;

struct FusedArgs {
  int Mrows, D, T, H, S, W, R;
  int kp_stride;       // entries per list (max(min(W, S), min(R, S)))
  int units;           // token blocks x 4H halves
  size_t sel_per_warp; // bytes of one selecting warp's region
  size_t sel_keys_bytes;
  int sel_kpad;
  uint32_t* lists;     // [B*T][H][2][2][kp_stride]: (b, h, t, which, half)
  int* dev_err;
};

__device__ __forceinline__ void mma_bf16_f(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                           uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %3, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %4, p;\n}\n" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(accumulate), "r"(kIdescF)
      : "memory");
}

// 8 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_load8(uint32_t taddr, uint32_t (&r)[8]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void epi_barrier() {  // the four epilogue warps
  asm volatile("bar.sync 1, %0;" ::"n"(F_EPI_WARPS * 32) : "memory");
}

__global__ void __launch_bounds__(kThreads, 1)
    project_select_kernel(const __grid_constant__ CUtensorMap tmX,
                          const __grid_constant__ CUtensorMap tmW, FusedArgs a) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t ring = (raw + 1023u) & ~1023u;  // tiles on 1,024-byte swizzle atoms
  const uint32_t a_ring = ring, b_ring = ring + F_ASTAGES * F_A_BYTES;
  unsigned char* gen = smem_raw + (ring - raw) + F_ASTAGES * F_A_BYTES + F_BSTAGES * F_B_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(gen);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + F_NUM_BARS);
  volatile int* stop = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int* epi_ok = reinterpret_cast<int*>(tmem_slot + 2);   // [F_EPI_WARPS]
  uint16_t* staging = reinterpret_cast<uint16_t*>(gen + 256);  // [FG][S]
  unsigned char* selw = gen + 256 + size_t(FG) * a.S * 2;      // per selecting warp
  const int AF = 0, AE = F_ASTAGES, BF = 2 * F_ASTAGES, BE = 2 * F_ASTAGES + F_BSTAGES,
            ACC_FULL = 2 * F_ASTAGES + 2 * F_BSTAGES, TMEM_EMPTY = ACC_FULL + 1, DRAIN = ACC_FULL + 2;
  auto bar = [&](int i) { return smem_u32(bars + i); };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int S = a.S, MT = S / 128, KB = (a.D + BK - 1) / BK, halves = 4 * a.H;
  const uint32_t tmem_cols = MT * FT <= 32 ? 32u : uint32_t(MT * FT);

  if (threadIdx.x == 0) {
    for (int i = 0; i < F_ASTAGES; ++i) {
      mbar_init(bar(AF + i), 1);
      mbar_init(bar(AE + i), 1);
    }
    for (int i = 0; i < F_BSTAGES; ++i) {
      mbar_init(bar(BF + i), 1);
      mbar_init(bar(BE + i), 1);
    }
    mbar_init(bar(ACC_FULL), 1);
    mbar_init(bar(TMEM_EMPTY), F_EPI_WARPS);
    mbar_init(bar(DRAIN), 1);
    *stop = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmX)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmW)) : "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_slot)),
                 "r"(tmem_cols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  // Producer: per stage, ever loaded / parity of its last load (read again after a stop).
  uint32_t a_used = 0, a_par = 0, b_used = 0, b_par = 0;
  if (warp == 0) {
    if (lane == 0) {
      // ---- TMA producer: per K step the X tile, then the MT W tiles ----
      int as = 0, bs = 0;
      uint32_t aph = 0, bph = 0;
      bool ok = true;
      for (int u = blockIdx.x; ok && u < a.units; u += gridDim.x) {
        const int tb = u / halves, g = u - tb * halves;
        for (int kb = 0; ok && kb < KB; ++kb) {
          if (!mbar_wait(bar(BE + bs), bph ^ 1u, stop)) {
            ok = false;
            break;
          }
          mbar_expect_tx(bar(BF + bs), F_B_BYTES);
          tma_load_2d(b_ring + uint32_t(bs) * F_B_BYTES, &tmX, kb * BK, tb * FT, bar(BF + bs));
          b_used |= 1u << bs;
          b_par = (b_par & ~(1u << bs)) | (bph << bs);
          if (++bs == F_BSTAGES) {
            bs = 0;
            bph ^= 1u;
          }
          for (int mt = 0; mt < MT; ++mt) {
            if (!mbar_wait(bar(AE + as), aph ^ 1u, stop)) {
              ok = false;
              break;
            }
            mbar_expect_tx(bar(AF + as), F_A_BYTES);
            tma_load_2d(a_ring + uint32_t(as) * F_A_BYTES, &tmW, kb * BK, g * S + mt * 128, bar(AF + as));
            a_used |= 1u << as;
            a_par = (a_par & ~(1u << as)) | (aph << as);
            if (++as == F_ASTAGES) {
              as = 0;
              aph ^= 1u;
            }
          }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---- MMA issuer ----
      int as = 0, bs = 0, it = 0;
      uint32_t aph = 0, bph = 0;
      bool ok = true;
      for (int u = blockIdx.x; ok && u < a.units; u += gridDim.x, ++it) {
        if (!mbar_wait(bar(TMEM_EMPTY), (uint32_t(it) & 1u) ^ 1u, stop)) break;
        tc_fence_after();
        for (int kb = 0; ok && kb < KB; ++kb) {
          if (!mbar_wait(bar(BF + bs), bph, stop)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sb = b_ring + uint32_t(bs) * F_B_BYTES;
          for (int mt = 0; mt < MT; ++mt) {
            if (!mbar_wait(bar(AF + as), aph, stop)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t sa = a_ring + uint32_t(as) * F_A_BYTES;
            const uint32_t d = tmem_base + uint32_t(mt * FT);
#pragma unroll
            for (int kk = 0; kk < BK / 16; ++kk)
              mma_bf16_f(d, sw128_desc(sa + kk * 32), sw128_desc(sb + kk * 32), (kb | kk) != 0);
            mma_commit(bar(AE + as));
            if (++as == F_ASTAGES) {
              as = 0;
              aph ^= 1u;
            }
          }
          if (!ok) break;
          mma_commit(bar(BE + bs));
          if (++bs == F_BSTAGES) {
            bs = 0;
            bph ^= 1u;
          }
        }
        if (ok) mma_commit(bar(ACC_FULL));
      }
      mma_commit(bar(DRAIN));
      mbar_wait_teardown(bar(DRAIN), 0);
    }
  } else {
    // ---- epilogue and selection: warp q reads TMEM lanes 32q .. 32q+31 ----
    const int q = warp & 3;         // TMEM lane quadrant of this warp
    const int sw = warp - 2;        // 0..3: this warp's selecting slot
    const CountSmem m = count_smem(selw + a.sel_per_warp * sw, a.sel_keys_bytes, a.sel_kpad,
                                   a.kp_stride);
    int it = 0;
    for (int u = blockIdx.x; u < a.units; u += gridDim.x, ++it) {
      // The four warps agree on whether the accumulators are ready (each waits; any that gave
      // up makes all leave), so no warp is left behind at a named barrier.
      const bool got = __all_sync(0xFFFFFFFFu, mbar_wait(bar(ACC_FULL), uint32_t(it) & 1u, stop));
      if (lane == 0) epi_ok[sw] = got ? 1 : 0;
      epi_barrier();
      const bool all = epi_ok[0] && epi_ok[1] && epi_ok[2] && epi_ok[3];
      epi_barrier();
      if (!all) break;
      tc_fence_after();
      const int tb = u / halves, g = u - tb * halves;
      const int which = g / (2 * a.H), h = (g >> 1) % a.H, half = g & 1;
      const int kin = min(which ? a.R : a.W, S);
#pragma unroll 1
      for (int grp = 0; grp < FT / FG; ++grp) {
        // tokens grp*8 .. grp*8+7 of the block: this warp's 32 sub-scores of every M-tile
#pragma unroll 1
        for (int mt = 0; mt < MT; ++mt) {
          uint32_t r[8];
          tmem_load8(tmem_base + (uint32_t(q * 32) << 16) + uint32_t(mt * FT + grp * FG), r);
          const int col = mt * 128 + q * 32 + lane;
#pragma unroll
          for (int n = 0; n < FG; ++n) {
            const __nv_bfloat16 v = __float2bfloat16_rn(__uint_as_float(r[n]));
            staging[n * S + col] = *reinterpret_cast<const uint16_t*>(&v);
          }
        }
        epi_barrier();
#pragma unroll 1
        for (int n = sw; n < FG; n += F_EPI_WARPS) {
          const int mrow = tb * FT + grp * FG + n;  // token b*T + t
          if (mrow < a.Mrows) {
            const uint16_t* row = staging + n * S;
            uint32_t* lst = m.la;
            if (!inner_count_smem(row, S, kin, m, lst)) inner_general_smem(row, S, kin, m, lst);
            const int b = mrow / a.T, t = mrow - b * a.T;
            uint32_t* dst = a.lists + ((((size_t(b) * a.H + h) * a.T + t) * 2 + which) * 2 + half) *
                                          size_t(a.kp_stride);
            for (int i = lane; i < kin; i += 32) dst[i] = lst[i];
            __syncwarp();
          }
        }
        epi_barrier();  // the staging buffer is free again
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(TMEM_EMPTY));
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                 "r"(tmem_cols)
                 : "memory");
  // After a stop, whichever role raised it, every copy issued lands before the CTA's shared
  // memory goes away.
  if (warp == 0 && lane == 0 && *stop) {
    for (int i = 0; i < F_ASTAGES; ++i)
      if (a_used & (1u << i)) mbar_wait_teardown(bar(AF + i), (a_par >> i) & 1u);
    for (int i = 0; i < F_BSTAGES; ++i)
      if (b_used & (1u << i)) mbar_wait_teardown(bar(BF + i), (b_par >> i) & 1u);
  }
  if (threadIdx.x == 0 && *stop && a.dev_err) atomicOr(a.dev_err, SDM_DEV_TIMEOUT);
}

// Outer top-K of every (b, h, t, k' or q') task from the inner lists (one warp per task).
struct OuterArgs {
  const uint32_t* lists;
  long long items;  // B * H * T
  int S, W, R, kp_stride;
  int cnt_w, cnt_r, kpad, warps;
  size_t per_warp, keys_bytes;
  const uint32_t* stair;  // both staircases (write, then read)
  int32_t* idx_w;
  float* sc_w;
  int32_t* idx_r;
  float* sc_r;
};

__global__ void __launch_bounds__(128, 6) outer_kernel(OuterArgs a) {
  extern __shared__ __align__(16) unsigned char smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long task = (long long)blockIdx.x * a.warps + warp;
  if (task >= 2 * a.items) return;
  const CountSmem m = count_smem(smem + a.per_warp * warp, a.keys_bytes, a.kpad, a.kp_stride);
  const int which = int(task & 1);
  const long long item = task >> 1;  // (b * H + h) * T + t
  const int K = which ? a.R : a.W, kin = min(K, a.S);
  const uint32_t* src = a.lists + (size_t(item) * 2 + which) * 2 * size_t(a.kp_stride);
  for (int i = lane; i < kin; i += 32) {
    m.la[i] = src[i];
    m.lb[i] = src[a.kp_stride + i];
  }
  __syncwarp();
  outer_task(m, which ? a.stair + a.cnt_w : a.stair, which ? a.cnt_r : a.cnt_w, K, kin, a.S,
             a.kpad, (which ? a.idx_r : a.idx_w) + item * K, (which ? a.sc_r : a.sc_w) + item * K);
}

// Bytes of the lists region of the fused projection's workspace.
size_t fused_lists_bytes(int B, int T, int H, int S, int W, int R) {
  const size_t kp = size_t(max(min(W, S), min(R, S)));
  return (size_t(B) * T * H * 4 * kp * 4 + 255) / 256 * 256;
}

}  // namespace

int launch_project(const void* x, const void* w, int B, int T, int D, int H, int S, void* kp,
                   void* qp, int* dev_err, int max_ctas, int pair, cudaStream_t s,
                   const ProjectStall* stall) {
  const long long Mrows = 1LL * B * T, Ncols = 4LL * H * S;
  if (Mrows == 0) return SDM_OK;
  const long long MT = (Mrows + BM - 1) / BM, NT = (Ncols + BN - 1) / BN;
  if (MT * NT > 0x7FFFFFFFLL || Mrows > 0x7FFFFFFFLL - 2 * BM) return SDM_EUNSUPPORTED;
  ProjArgs pa;
  pa.Mrows = int(Mrows);
  pa.Ncols = int(Ncols);
  pa.D = D;
  pa.T = T;
  pa.H = H;
  pa.S = S;
  pa.kp = static_cast<uint16_t*>(kp);
  pa.qp = static_cast<uint16_t*>(qp);
  pa.dev_err = dev_err;
  pa.wait_ns = stall ? stall->wait_ns : kWaitNs;
  pa.stall_cta = stall ? stall->cta : -1;
  pa.stall_step = stall ? stall->step : 0;
  CUtensorMap tmX, tmW;
  if (!bf16_tile_map(&tmX, x, int(Mrows), D, BM) || !bf16_tile_map(&tmW, w, int(Ncols), D, BN / 2))
    return SDM_ECUDA;
  const int mode = pair < 0 ? (MT >= 2 ? 2 : 0) : pair;  // 0 single CTAs, 2 2-SM MMA pairs
  if (mode != 0 && mode != 2) return SDM_EINVAL;
  const int CL = mode == 0 ? 1 : 2;
  const long long units = ((MT + CL - 1) / CL) * NT;
  const bool vec = (2 * S) % 8 == 0 && aligned16(kp) && aligned16(qp);
  const void* fn = mode == 2 ? (vec ? reinterpret_cast<const void*>(&project_kernel_2sm<true>)
                                    : reinterpret_cast<const void*>(&project_kernel_2sm<false>))
                             : (vec ? reinterpret_cast<const void*>(&project_kernel<true>)
                                    : reinterpret_cast<const void*>(&project_kernel<false>));
  const int smem = mode == 2 ? kSmemBytes2 : kSmemBytes;
  if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
    return SDM_ECUDA;
  const int sms = sm_count();
  if (sms <= 0) return SDM_ECUDA;
  long long clusters = sms / CL;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = unsigned(CL);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(clusters * CL));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = size_t(smem);
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (CL > 1) {  // a persistent grid larger than what can be resident would run in two waves
    int active = 0;
    if (cudaOccupancyMaxActiveClusters(&active, fn, &cfg) != cudaSuccess || active <= 0)
      return SDM_ECUDA;
    if (active < clusters) clusters = active;
  }
  if (max_ctas > 0 && max_ctas / CL < clusters) clusters = max_ctas / CL > 0 ? max_ctas / CL : 1;
  if (units < clusters) clusters = units;
  cfg.gridDim = dim3(unsigned(clusters * CL));
  void* args[] = {&tmX, &tmW, &pa};
  if (cudaLaunchKernelExC(&cfg, fn, args) != cudaSuccess) return SDM_ECUDA;
  return last_launch_status();
}

size_t project_select_workspace(int B, int T, int H, int S, int W, int R) {
  return fused_lists_bytes(B, T, H, S, W, R) +
         (size_t(stair_table_words(W, R, S)) * 4 + 255) / 256 * 256;
}

int launch_project_select(const void* x, const void* w, int B, int T, int D, int H, int S, int W,
                          int R, int32_t* idx_w, float* sc_w, int32_t* idx_r, float* sc_r,
                          void* workspace, int* dev_err, cudaStream_t s) {
  const long long Mrows = 1LL * B * T;
  if (Mrows == 0) return SDM_OK;
  if (S % 128 || S > kCountMaxS || W > kCountMaxK || R > kCountMaxK) return SDM_EUNSUPPORTED;
  const long long blocks_t = (Mrows + FT - 1) / FT;
  if (blocks_t * 4 * H > 0x7FFFFFFFLL || Mrows > 0x7FFFFFFFLL - FT) return SDM_EUNSUPPORTED;
  FusedArgs fa;
  fa.Mrows = int(Mrows);
  fa.D = D;
  fa.T = T;
  fa.H = H;
  fa.S = S;
  fa.W = W;
  fa.R = R;
  fa.kp_stride = max(min(W, S), min(R, S));
  fa.units = int(blocks_t * 4 * H);
  fa.sel_kpad = 32;
  while (fa.sel_kpad < max(W, R)) fa.sel_kpad <<= 1;
  fa.sel_keys_bytes = (size_t(S) * 4 + 15) / 16 * 16;
  fa.sel_per_warp = (count_per_warp_bytes(fa.sel_keys_bytes, fa.sel_kpad, fa.kp_stride) + 15) / 16 * 16;
  fa.lists = static_cast<uint32_t*>(workspace);
  fa.dev_err = dev_err;
  CUtensorMap tmX, tmW;
  if (!bf16_tile_map(&tmX, x, int(Mrows), D, FT) || !bf16_tile_map(&tmW, w, 4 * H * S, D, 128))
    return SDM_ECUDA;
  const size_t smem = size_t(F_ASTAGES) * F_A_BYTES + size_t(F_BSTAGES) * F_B_BYTES + 1024 + 256 +
                      size_t(FG) * S * 2 + size_t(F_EPI_WARPS) * fa.sel_per_warp;
  int dev = 0, max_smem = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
    return SDM_ECUDA;
  if (smem > size_t(max_smem)) return SDM_EUNSUPPORTED;
  const void* fn = reinterpret_cast<const void*>(&project_select_kernel);
  if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)) != cudaSuccess)
    return SDM_ECUDA;
  const int sms = sm_count();
  if (sms <= 0) return SDM_ECUDA;
  const int grid = fa.units < sms ? fa.units : sms;
  void* args[] = {&tmX, &tmW, &fa};
  if (cudaLaunchKernel(fn, dim3(unsigned(grid)), dim3(kThreads), args, smem, s) != cudaSuccess)
    return SDM_ECUDA;
  if (last_launch_status() != SDM_OK) return SDM_ECUDA;

  // The outer top-K from the lists, with both staircases in the workspace after them.
  uint32_t* stair = reinterpret_cast<uint32_t*>(static_cast<unsigned char*>(workspace) +
                                                fused_lists_bytes(B, T, H, S, W, R));
  int st = launch_stair_table(stair, W, R, S, s);
  if (st != SDM_OK) return st;
  OuterArgs oa;
  oa.lists = fa.lists;
  oa.items = Mrows * H;
  oa.S = S;
  oa.W = W;
  oa.R = R;
  oa.kp_stride = fa.kp_stride;
  oa.cnt_w = stair_count(W, min(W, S));
  oa.cnt_r = stair_count(R, min(R, S));
  oa.kpad = fa.sel_kpad;
  oa.warps = 4;
  oa.keys_bytes = select_key_bytes(oa.kpad, S, max(oa.cnt_w, oa.cnt_r), 4);
  oa.per_warp = (count_per_warp_bytes(oa.keys_bytes, oa.kpad, oa.kp_stride) + 15) / 16 * 16;
  oa.stair = stair;
  oa.idx_w = idx_w;
  oa.sc_w = sc_w;
  oa.idx_r = idx_r;
  oa.sc_r = sc_r;
  const size_t osmem = oa.per_warp * oa.warps;
  const void* ofn = reinterpret_cast<const void*>(&outer_kernel);
  if (cudaFuncSetAttribute(ofn, cudaFuncAttributeMaxDynamicSharedMemorySize, int(osmem)) != cudaSuccess ||
      cudaFuncSetAttribute(ofn, cudaFuncAttributePreferredSharedMemoryCarveout,
                           int(cudaSharedmemCarveoutMaxShared)) != cudaSuccess)
    return SDM_ECUDA;
  const long long oblocks = (2 * oa.items + oa.warps - 1) / oa.warps;
  if (oblocks > 0x7FFFFFFFLL) return SDM_EUNSUPPORTED;
  void* oargs[] = {&oa};
  if (cudaLaunchKernel(ofn, dim3(unsigned(oblocks)), dim3(oa.warps * 32), oargs, osmem, s) != cudaSuccess)
    return SDM_ECUDA;
  return last_launch_status();
}

int launch_bounded_wait(int mode, unsigned long long limit_ns, int* dev_err,
                        unsigned long long* elapsed_ns, cudaStream_t s) {
  bounded_wait_kernel<<<1, 32, 0, s>>>(mode, limit_ns, dev_err, elapsed_ns);
  return last_launch_status();
}

}  // namespace sdm
