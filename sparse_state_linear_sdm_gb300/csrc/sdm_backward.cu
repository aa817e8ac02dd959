// Backward pass of the sparse gated-delta scan (Sparse Delta Memory technical summary,
// gist.science/it/paper/2607.07386, "Meccanismo Core" items 2-4; the learned initial state
// of "Stato Iniziale Appreso" receives dL/dM_0).  Reverse mode for the loss
// L = sum_t <dO_t, o_t> + <dM_T, M_T>, with the selected slots held fixed (they are
// discrete).  The forward (sdm_scan_forward_train) keeps, per token, the write rows before
// their update (w_prev) and the read rows as read (r_rows); the backward walks the tokens
// from last to first with the adjoint G = dL/dM_t, a table like M:
//   read   o_t = sum_j r_j M_t[ir_j]:  G[ir_j] += r_j dO_t,  dr_j = <dO_t, M_t[ir_j]>
//   write  M_t[i] = a M_{t-1}[i] + b k_i (v_t - a M_{t-1}[i]), with G after the read:
//          dv_t += b k_i G[i],  ge_i = <G[i], v_t - a M_{t-1}[i]>,  gm_i = <G[i], M_{t-1}[i]>,
//          then G[i] <- a (1 - b k_i) G[i]
//   finish dk_i = b ge_i,  da_t = sum_i (1 - b k_i) gm_i,  db_t = sum_i k_i ge_i, and the
//          softmax backward ds_i = w_i (dw_i - sum_l w_l dw_l) for the write and read scores.
//
// Kernels: the reverse scan (one block per (b, h, slice of columns), sequential in t; the
// dot products over d_v leave one partial per slice), a finish kernel (one warp per token:
// sums the slices' partials, softmax backward), a batch reduction of G into dM_0, and the
// selection backward (a selected score is half0[i] + half1[j]).
//
// Zero final adjoint (SDM_BWD_FINAL_ZERO, dL/dM_T = 0, the usual training loss on the
// outputs alone).  Going backwards, a row's adjoint stays exactly zero until a read of the
// row adds r_j dO_t; a write only scales it.  So the adjoint row seen at a slot is zero iff
// no read of that row comes later in the forward order (a read at the same token comes
// after the token's writes).  Two passes find this before the reverse scan: the last token
// that reads each row (an atomic maximum per read slot into a per-(b, h) table), then one
// bit per slot.  The reverse scan then skips, at a zero slot, the adjoint load and, for a
// write slot, the stored row's load and the adjoint store (the row stays zero); every
// non-zero row it loads was stored earlier in the same pass.  G's contents on entry are
// never read; the batch reduction writes zeros to the rows no slot reads.  Every product
// and sum that remains is the one the full pass forms, and the skipped terms are exact
// zeros, so the outputs equal the full pass's with G cleared (up to the sign of zeros).
#include "sdm_internal.cuh"

namespace sdm {
namespace {

constexpr int kBwdThreads = 256;
constexpr int kBwdWarps = kBwdThreads / 32;

struct BwdArgs {
  const int32_t* idx_w;
  const float* sc_w;
  const int32_t* idx_r;
  const float* sc_r;
  const void* v;
  int v_bf16;
  const float* alpha;
  const float* beta;
  const float* w_prev;
  const float* r_rows;
  const float* dO;
  float* G;
  float* dv;
  float* part;  // [BH, T, slices, 2W + R]: ge (W), gm (W), dr (R) of one column slice
  const float* wts;  // [BH, T, W + R]: softmax of the write, then of the read scores
  // [BH, T, NW + NS] per token: NW words, bit e = slot e of [write | read] sees a zero
  // adjoint (all 0 unless dL/dM_T = 0); then NS words, bit i = write slot i's row is also a
  // read slot of the same token (its adjoint is the read phase's update: loaded after it).
  const uint32_t* flags;
  int NW, NS, NF;  // NF: words per token, NW + NS padded to a multiple of 4
  bool zero_final;
  bool vec16;  // W, R multiples of 4 and the slot arrays 16-byte aligned: 16-byte staging
  int T;
  long long N;
  int d_v, W, R;
};

__device__ __forceinline__ float4 load_v4(const void* v, int bf16, size_t i4) {
  if (bf16) {
    const uint2 u = reinterpret_cast<const uint2*>(v)[i4];
    return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xFFFF0000u),
                       __uint_as_float(u.y << 16), __uint_as_float(u.y & 0xFFFF0000u));
  }
  return reinterpret_cast<const float4*>(v)[i4];
}

__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gmem_src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(
                   static_cast<uint32_t>(__cvta_generic_to_shared(smem_dst))),
               "l"(gmem_src)
               : "memory");
}

__device__ __forceinline__ float dot4(float4 a, float4 b) {
  return fmaf(a.w, b.w, fmaf(a.z, b.z, fmaf(a.y, b.y, a.x * b.x)));
}

// Sum over the LPR lanes that hold one row slice (lanes differing in the low bits).
template <int LPR>
__device__ __forceinline__ float slice_sum(float x) {
#pragma unroll
  for (int off = 1; off < LPR; off <<= 1) x += __shfl_xor_sync(0xFFFFFFFFu, x, off);
  return x;
}

template <int C>
__global__ void __launch_bounds__(kBwdThreads) scan_backward_kernel(BwdArgs a) {
  constexpr int LPR = C / 4;                 // threads per row slice (one float4 each)
  constexpr int RPP = kBwdThreads / LPR;     // row slices per pass
  constexpr int NB = 4;                      // rows per thread per round, loaded together
  extern __shared__ __align__(16) unsigned char smem[];
  const int W = a.W, R = a.R, T = a.T, d_v = a.d_v;
  const int WR = W + R;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  float* red = reinterpret_cast<float*>(smem);  // [2][warps][C], by token parity
  // Two staging buffers of one token's [slots W | slots R | weights W | weights R | zero
  // bits] (the weights from the softmax pass): the next token's (going backwards) arrive by
  // cp.async while this one is processed.
  const int NF = a.NF;
  const int SB = 2 * WR + NF;
  int32_t* stg = reinterpret_cast<int32_t*>(red + 2 * kBwdWarps * C);  // [2][SB]

  const int slices = d_v / C;
  const int bh = blockIdx.x / slices;
  const int sl = blockIdx.x - bh * slices;
  const int c0 = sl * C;
  const int c4 = tid % LPR;
  const int PW = 2 * W + R;
  float* Gbh = a.G + size_t(bh) * size_t(a.N) * d_v + c0;

  auto stage = [&](int t) {  // into buffer t & 1
    const size_t tk = size_t(bh) * T + t;
    int32_t* dst = stg + (t & 1) * SB;
    if (a.vec16) {  // the four segments are contiguous per token: 16-byte copies
      const int n1 = W / 4, n2 = n1 + R / 4, n3 = n2 + WR / 4, n4 = n3 + NF / 4;
      for (int q = tid; q < n4; q += kBwdThreads) {
        const void* src = q < n1 ? static_cast<const void*>(a.idx_w + tk * W + 4 * q)
                        : q < n2 ? static_cast<const void*>(a.idx_r + tk * R + 4 * (q - n1))
                        : q < n3 ? static_cast<const void*>(a.wts + tk * WR + 4 * (q - n2))
                                 : static_cast<const void*>(a.flags + tk * NF + 4 * (q - n3));
        cp_async16(dst + 4 * q, src);
      }
      asm volatile("cp.async.commit_group;" ::: "memory");
      return;
    }
    for (int e = tid; e < SB; e += kBwdThreads) {
      const void* src = e < W ? static_cast<const void*>(a.idx_w + tk * W + e)
                      : e < WR ? static_cast<const void*>(a.idx_r + tk * R + (e - W))
                      : e < 2 * WR ? static_cast<const void*>(a.wts + tk * WR + (e - WR))
                                   : static_cast<const void*>(a.flags + tk * NF + (e - 2 * WR));
      asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(
                       static_cast<uint32_t>(__cvta_generic_to_shared(dst + e))),
                   "l"(src)
                   : "memory");
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
  };
  if (T > 0) stage(T - 1);
  asm volatile("cp.async.wait_all;" ::: "memory");
  __syncthreads();

  for (int t = T - 1; t >= 0; --t) {
    const size_t tk = size_t(bh) * T + t;
    const int32_t* iw = stg + (t & 1) * SB;
    const int32_t* ir = iw + W;
    const float* kw = reinterpret_cast<const float*>(iw + WR);  // the token's write weights
    const float* rw = kw + W;                                    // and read weights
    const uint32_t* zb = reinterpret_cast<const uint32_t*>(iw + 2 * WR);
    const uint32_t* sb = zb + a.NW;
    auto zero_at = [&](int e) { return a.zero_final && ((zb[e >> 5] >> (e & 31)) & 1u) != 0; };
    auto same_at = [&](int i) { return ((sb[i >> 5] >> (i & 31)) & 1u) != 0; };
    if (t > 0) stage(t - 1);  // the other buffer held token t+1, retired at its last barrier
    float* part = a.part + (tk * slices + sl) * PW;

    // The write phase's first round of rows, loaded now so that their latency overlaps the
    // read phase's: a write row's adjoint depends on this token's reads only when one of its
    // read slots names the same row (marked by the flags pass; loaded after the barrier).
    // A zero adjoint row contributes nothing and stays zero: no loads, no store.
    int32_t xw[NB];
    float4 g0[NB], wp0[NB];
    bool late[NB];
#pragma unroll
    for (int u = 0; u < NB; ++u) {
      const int i = u * RPP + tid / LPR;
      xw[u] = i < W ? iw[i] : -1;
      if (xw[u] >= 0 && xw[u] < a.N && zero_at(i)) xw[u] = -1;
      const bool ok = xw[u] >= 0 && xw[u] < a.N;
      late[u] = ok && same_at(i);
      g0[u] = wp0[u] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (ok) {
        if (!late[u]) g0[u] = reinterpret_cast<const float4*>(Gbh + size_t(xw[u]) * d_v)[c4];
        wp0[u] = reinterpret_cast<const float4*>(a.w_prev + (tk * W + i) * d_v + c0)[c4];
      }
    }
    const float4 dO4 = reinterpret_cast<const float4*>(a.dO + tk * d_v + c0)[c4];

    // Read rows: dr_j (this slice's share) and G[ir_j] += r_j dO_t.  Each thread takes up
    // to NB rows per round and loads all of them before using any (their latencies
    // overlap); the round bound is the same for every lane (the shuffles need the whole
    // warp), `in` marks real rows.
    for (int jb = 0; jb < R; jb += NB * RPP) {
      int32_t x[NB];
      float4 gv[NB], m[NB];
#pragma unroll
      for (int u = 0; u < NB; ++u) {
        const int j = jb + u * RPP + tid / LPR;
        x[u] = j < R ? ir[j] : -1;
        const bool ok = x[u] >= 0 && x[u] < a.N;  // uniform over the row's LPR lanes
        gv[u] = m[u] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (ok) {
          if (!zero_at(W + j)) gv[u] = reinterpret_cast<const float4*>(Gbh + size_t(x[u]) * d_v)[c4];
          m[u] = reinterpret_cast<const float4*>(a.r_rows + (tk * R + j) * d_v + c0)[c4];
        }
      }
#pragma unroll
      for (int u = 0; u < NB; ++u) {
        const int j = jb + u * RPP + tid / LPR;
        const float s = slice_sum<LPR>(dot4(dO4, m[u]));
        if (j < R && c4 == 0) part[2 * W + j] = s;
        if (x[u] >= 0 && x[u] < a.N) {
          const float r = rw[j];
          reinterpret_cast<float4*>(Gbh + size_t(x[u]) * d_v)[c4] =
              make_float4(fmaf(r, dO4.x, gv[u].x), fmaf(r, dO4.y, gv[u].y), fmaf(r, dO4.z, gv[u].z),
                          fmaf(r, dO4.w, gv[u].w));
        }
      }
    }
    __syncthreads();  // the read contributions reach G before the write rows load it

    // Write rows: partial dot products, dv, and G propagated to M_{t-1} (same batching).
    const float al = a.alpha[tk], be = a.beta[tk];
    const float4 vv = load_v4(a.v, a.v_bf16, (tk * d_v + c0) / 4 + c4);
    float4 dva = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int ib = 0; ib < W; ib += NB * RPP) {
      int32_t x[NB];
      float4 g[NB], wp[NB];
      if (ib == 0) {
#pragma unroll
        for (int u = 0; u < NB; ++u) {
          x[u] = xw[u];
          g[u] = late[u] ? reinterpret_cast<const float4*>(Gbh + size_t(xw[u]) * d_v)[c4] : g0[u];
          wp[u] = wp0[u];
        }
      } else {
#pragma unroll
        for (int u = 0; u < NB; ++u) {
          const int i = ib + u * RPP + tid / LPR;
          x[u] = i < W ? iw[i] : -1;
          if (x[u] >= 0 && x[u] < a.N && zero_at(i)) x[u] = -1;
          g[u] = wp[u] = make_float4(0.f, 0.f, 0.f, 0.f);
          if (x[u] >= 0 && x[u] < a.N) {
            g[u] = reinterpret_cast<const float4*>(Gbh + size_t(x[u]) * d_v)[c4];
            wp[u] = reinterpret_cast<const float4*>(a.w_prev + (tk * W + i) * d_v + c0)[c4];
          }
        }
      }
#pragma unroll
      for (int u = 0; u < NB; ++u) {
        const int i = ib + u * RPP + tid / LPR;
        const bool in = i < W;
        const float4 e = make_float4(fmaf(-al, wp[u].x, vv.x), fmaf(-al, wp[u].y, vv.y),
                                     fmaf(-al, wp[u].z, vv.z), fmaf(-al, wp[u].w, vv.w));
        const float ge = slice_sum<LPR>(dot4(g[u], e));
        const float gm = slice_sum<LPR>(dot4(g[u], wp[u]));
        if (in && c4 == 0) {
          part[i] = ge;
          part[W + i] = gm;
        }
        const float bk = in ? be * kw[i] : 0.f;
        dva.x = fmaf(bk, g[u].x, dva.x);
        dva.y = fmaf(bk, g[u].y, dva.y);
        dva.z = fmaf(bk, g[u].z, dva.z);
        dva.w = fmaf(bk, g[u].w, dva.w);
        if (x[u] >= 0 && x[u] < a.N) {
          const float sc = al * (1.f - bk);
          reinterpret_cast<float4*>(Gbh + size_t(x[u]) * d_v)[c4] =
              make_float4(sc * g[u].x, sc * g[u].y, sc * g[u].z, sc * g[u].w);
        }
      }
    }
    // dv_t: sum over the rows held by the other lanes and warps.
#pragma unroll
    for (int off = LPR; off < 32; off <<= 1) {
      dva.x += __shfl_xor_sync(0xFFFFFFFFu, dva.x, off);
      dva.y += __shfl_xor_sync(0xFFFFFFFFu, dva.y, off);
      dva.z += __shfl_xor_sync(0xFFFFFFFFu, dva.z, off);
      dva.w += __shfl_xor_sync(0xFFFFFFFFu, dva.w, off);
    }
    float* rd = red + (t & 1) * kBwdWarps * C;
    if (lane < LPR) reinterpret_cast<float4*>(rd + warp * C)[lane] = dva;
    asm volatile("cp.async.wait_all;" ::: "memory");
    // G of this token is written before the previous token loads it; the next token's slots
    // and scores and this token's dv partials are visible.
    __syncthreads();
    if (tid < LPR) {
      float4 s4 = reinterpret_cast<const float4*>(rd)[tid];
      for (int w = 1; w < kBwdWarps; ++w) {
        const float4 u = reinterpret_cast<const float4*>(rd + w * C)[tid];
        s4 = make_float4(s4.x + u.x, s4.y + u.y, s4.z + u.z, s4.w + u.w);
      }
      reinterpret_cast<float4*>(a.dv + tk * d_v + c0)[tid] = s4;
    }
  }
}

size_t backward_smem_bytes(int C, int W, int R, int NF) {
  return size_t(2 * kBwdWarps) * C * 4 + size_t(2 * (2 * (W + R) + NF)) * 4;
}

// Softmax of every token's write and read scores, one warp per (b, h, t), with the routine
// the planning kernel and the finish kernel use: the reverse scan stages these weights with
// the slots instead of forming them on its sequential path.
__global__ void __launch_bounds__(256) bwd_weights_kernel(const float* __restrict__ sc_w,
                                                          const float* __restrict__ sc_r, int W,
                                                          int R, long long tokens,
                                                          float* __restrict__ wts) {
  const long long tok = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (tok >= tokens) return;
  float* out = wts + tok * (W + R);
  warp_softmax(sc_w + tok * W, W, out);
  warp_softmax(sc_r + tok * R, R, out + W);
}

// --- zero final adjoint: which slots see a zero adjoint row ---------------------------

// One warp per (b, h, t): last[bh][x] = max(last[bh][x], t) for every read slot x.
__global__ void __launch_bounds__(256) last_read_kernel(const int32_t* __restrict__ idx_r, int T,
                                                        int R, long long N, long long tokens,
                                                        int32_t* __restrict__ last) {
  const long long tok = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (tok >= tokens) return;
  const long long bh = tok / T;
  const int t = int(tok - bh * T);
  int32_t* lb = last + bh * N;
  for (int j = threadIdx.x & 31; j < R; j += 32) {
    const int32_t x = idx_r[tok * R + j];
    if (x >= 0 && x < N) atomicMax(lb + x, t);
  }
}

// One warp per (b, h, t).  Zero bits (when last is given, dL/dM_T = 0): bit e of the
// token's [write | read] slots is set when the adjoint row at that slot is zero: a write
// slot whose row no read at token >= t selects, a read slot whose row no read after t
// selects.  Same-token bits: bit i when write slot i's row is also one of the token's read
// slots (through a hash of the read slots in the warp's shared memory, at most half full).
// Slots outside [0, N) get 0.
__global__ void __launch_bounds__(256) bwd_flags_kernel(const int32_t* __restrict__ idx_w,
                                                        const int32_t* __restrict__ idx_r, int T,
                                                        int W, int R, long long N, long long tokens,
                                                        const int32_t* __restrict__ last, int NW,
                                                        int NS, int NF, int log2cap,
                                                        uint32_t* __restrict__ flags) {
  extern __shared__ int32_t tabs[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long tok = (long long)blockIdx.x * (blockDim.x >> 5) + warp;
  if (tok >= tokens) return;
  const int cap = 1 << log2cap;
  int32_t* tab = tabs + size_t(warp) * cap;
  const long long bh = tok / T;
  const int t = int(tok - bh * T);
  uint32_t* out = flags + tok * NF;
  auto hash = [&](int32_t x) { return (uint32_t(x) * 0x9E3779B1u) >> (32 - log2cap); };
  for (int i = lane; i < cap; i += 32) tab[i] = -1;
  __syncwarp();
  for (int j = lane; j < R; j += 32) {
    const int32_t x = idx_r[tok * R + j];
    if (x < 0 || x >= N) continue;
    for (uint32_t h = hash(x);; h = (h + 1) & uint32_t(cap - 1)) {
      const int32_t prev = atomicCAS(&tab[h], -1, x);
      if (prev == -1 || prev == x) break;
    }
  }
  __syncwarp();
  const int32_t* lb = last ? last + bh * N : nullptr;
  for (int e0 = 0; e0 < W + R; e0 += 32) {
    const int e = e0 + lane;
    bool z = false;
    if (lb && e < W + R) {
      const int32_t x = e < W ? idx_w[tok * W + e] : idx_r[tok * R + (e - W)];
      if (x >= 0 && x < N) {
        const int32_t l = lb[x];
        z = e < W ? l < t : l == t;
      }
    }
    const unsigned m = __ballot_sync(0xFFFFFFFFu, z);
    if (lane == 0) out[e0 >> 5] = m;
  }
  for (int i0 = 0; i0 < W; i0 += 32) {
    const int i = i0 + lane;
    bool same = false;
    if (i < W) {
      const int32_t x = idx_w[tok * W + i];
      if (x >= 0 && x < N)
        for (uint32_t h = hash(x);; h = (h + 1) & uint32_t(cap - 1)) {
          const int32_t v = tab[h];
          if (v == -1) break;
          if (v == x) {
            same = true;
            break;
          }
        }
    }
    const unsigned m = __ballot_sync(0xFFFFFFFFu, same);
    if (lane == 0) out[NW + (i0 >> 5)] = m;
  }
}

int backward_cols(int d_v) {
  for (int c : {32, 16, 8, 4})
    if (d_v % c == 0) return c;
  return 0;
}

// One warp per (b, h, t): sums the slices' partials, then the softmax backward with the
// weights of the softmax pass (wts [items, W + R]).
__global__ void __launch_bounds__(128) backward_finish_kernel(
    const float* __restrict__ wts, const float* __restrict__ beta,
    const float* __restrict__ part, int slices, int W, int R, long long items, float* dalpha,
    float* dbeta, float* dsc_w, float* dsc_r) {
  extern __shared__ __align__(16) unsigned char smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float* k = reinterpret_cast<float*>(smem) + size_t(warp) * 2 * (W + R);
  float* r = k + W;
  float* dk = r + R;
  float* dr = dk + W;
  const long long item = (long long)blockIdx.x * (blockDim.x >> 5) + warp;
  if (item >= items) return;
  for (int i = lane; i < W + R; i += 32) k[i] = wts[item * (W + R) + i];  // k then r
  __syncwarp();
  const int PW = 2 * W + R;
  const float* p = part + item * slices * PW;
  const float be = beta[item];
  float sa = 0.f, sb = 0.f, dotk = 0.f;
  for (int i = lane; i < W; i += 32) {
    float ge = 0.f, gm = 0.f;
    for (int s = 0; s < slices; ++s) {
      ge += p[s * PW + i];
      gm += p[s * PW + W + i];
    }
    const float d = be * ge;
    dk[i] = d;
    dotk = fmaf(k[i], d, dotk);
    sa = fmaf(1.f - be * k[i], gm, sa);
    sb = fmaf(k[i], ge, sb);
  }
  float dotr = 0.f;
  for (int j = lane; j < R; j += 32) {
    float d = 0.f;
    for (int s = 0; s < slices; ++s) d += p[s * PW + 2 * W + j];
    dr[j] = d;
    dotr = fmaf(r[j], d, dotr);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    sa += __shfl_xor_sync(0xFFFFFFFFu, sa, off);
    sb += __shfl_xor_sync(0xFFFFFFFFu, sb, off);
    dotk += __shfl_xor_sync(0xFFFFFFFFu, dotk, off);
    dotr += __shfl_xor_sync(0xFFFFFFFFu, dotr, off);
  }
  __syncwarp();
  for (int i = lane; i < W; i += 32) dsc_w[item * W + i] = k[i] * (dk[i] - dotk);
  for (int j = lane; j < R; j += 32) dsc_r[item * R + j] = r[j] * (dr[j] - dotr);
  if (lane == 0) {
    dalpha[item] = sa;
    dbeta[item] = sb;
  }
}

// Zero final adjoint: rows that no read selects hold no adjoint (G was never written
// there), so they are set to zero, and dM0[h] (if given) = sum over the batch of G[b, h]
// with those rows taken as zero, in the batch order of reduce_batch_kernel.  One warp per
// group of 32 rows of (h, row): lane j first reads row j's table entry of every batch row
// (coalesced) into a bit mask, so that the G loads that follow depend on no other load;
// then the lanes cover the group's float4 pieces.  B <= 32 (the host takes the plain loop
// of reduce_batch_zero_wide_kernel beyond).
__global__ void __launch_bounds__(256) reduce_batch_zero_kernel(float4* __restrict__ G,
                                                                float4* __restrict__ dM0,
                                                                const int32_t* __restrict__ last,
                                                                int B, long long rows, int dv4,
                                                                bool write_zeros) {
  const long long warps = (long long)gridDim.x * (blockDim.x >> 5);
  const int lane = threadIdx.x & 31;
  const long long groups = (rows + 31) / 32;
  for (long long g = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); g < groups;
       g += warps) {
    const long long row0 = g * 32;
    const int nrows = int(min(32LL, rows - row0));
    uint32_t bits = 0;  // bit b: batch row b reads row row0 + lane
    if (lane < nrows)
      for (int b = 0; b < B; ++b)
        bits |= uint32_t(last[size_t(b) * size_t(rows) + size_t(row0 + lane)] >= 0) << b;
    for (int e0 = 0; e0 < 32 * dv4; e0 += 32) {
      const int e = e0 + lane, r = e / dv4, c = e - r * dv4;
      const uint32_t m = __shfl_sync(0xFFFFFFFFu, bits, r & 31);
      if (r >= nrows) continue;
      const size_t row = size_t(row0 + r);
      float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int b0 = 0; b0 < B; b0 += 8) {
        float4 u[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          u[k] = make_float4(0.f, 0.f, 0.f, 0.f);
          if (b0 + k < B && ((m >> (b0 + k)) & 1u)) u[k] = G[(size_t(b0 + k) * size_t(rows) + row) * dv4 + c];
        }
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const int b = b0 + k;
          if (b < B) {
            if (write_zeros && !((m >> b) & 1u)) __stcs(G + (size_t(b) * size_t(rows) + row) * dv4 + c, u[k]);
            s = b == 0 ? u[k] : make_float4(s.x + u[k].x, s.y + u[k].y, s.z + u[k].z, s.w + u[k].w);
          }
        }
      }
      if (dM0) dM0[row * dv4 + c] = s;
    }
  }
}

// The same for any B: one warp per (h, row), the table entry read before each load.
__global__ void __launch_bounds__(256) reduce_batch_zero_wide_kernel(float4* __restrict__ G,
                                                                     float4* __restrict__ dM0,
                                                                     const int32_t* __restrict__ last,
                                                                     int B, long long rows, int dv4,
                                                                     bool write_zeros) {
  const long long warps = (long long)gridDim.x * (blockDim.x >> 5);
  const int lane = threadIdx.x & 31;
  for (long long row = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); row < rows;
       row += warps) {
    for (int c = lane; c < dv4; c += 32) {
      float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int b = 0; b < B; ++b) {
        const size_t rb = size_t(b) * size_t(rows) + size_t(row);
        float4 u = make_float4(0.f, 0.f, 0.f, 0.f);
        if (last[rb] >= 0)
          u = G[rb * dv4 + c];
        else if (write_zeros)
          __stcs(G + rb * dv4 + c, u);
        s = b == 0 ? u : make_float4(s.x + u.x, s.y + u.y, s.z + u.z, s.w + u.w);
      }
      if (dM0) dM0[size_t(row) * dv4 + c] = s;
    }
  }
}

// dM0[h] = sum over the batch of G[b, h].
__global__ void reduce_batch_kernel(const float4* __restrict__ G, float4* __restrict__ dM0, int B,
                                    size_t per_batch4) {
  const size_t stride = size_t(gridDim.x) * blockDim.x;
  for (size_t i = size_t(blockIdx.x) * blockDim.x + threadIdx.x; i < per_batch4; i += stride) {
    float4 s = G[i];
    for (int b = 1; b < B; ++b) {
      const float4 u = G[size_t(b) * per_batch4 + i];
      s = make_float4(s.x + u.x, s.y + u.y, s.z + u.z, s.w + u.w);
    }
    dM0[i] = s;
  }
}

// Selection backward, one warp per (b, h, t): dhalves[0][i] and dhalves[1][j] collect the
// gradients of the selected scores that use them (flat = i * S + j).
__global__ void __launch_bounds__(128) select_backward_kernel(const int32_t* __restrict__ idx,
                                                              const float* __restrict__ dsc,
                                                              long long items, int S, int K,
                                                              float* dhalves) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long item = (long long)blockIdx.x * (blockDim.x >> 5) + warp;
  if (item >= items) return;
  float* dh = dhalves + item * 2 * S;
  for (int i = lane; i < 2 * S; i += 32) dh[i] = 0.f;
  __syncwarp();
  for (int r = lane; r < K; r += 32) {
    const int32_t f = idx[item * K + r];
    if (f < 0 || f >= S * S) continue;
    const float d = dsc[item * K + r];
    atomicAdd(dh + f / S, d);
    atomicAdd(dh + S + f % S, d);
  }
}

// Workspace of the reverse pass: [part | weights | last-read table | zero bits], each piece
// 16-byte aligned; the last two only with SDM_BWD_FINAL_ZERO.  0 on overflow or bad sizes.
struct BwdWorkspace {
  size_t part, wts, flags, last, total;
};

// Flag words per token (zero bits, then same-token bits), padded to 16 bytes.
inline int bwd_flag_words(int W, int R) {
  return ((W + R + 31) / 32 + (W + 31) / 32 + 3) & ~3;
}

bool backward_workspace(int B, int H, int T, long long N, int d_v, int W, int R, unsigned flags,
                        BwdWorkspace* ws) {
  if (B < 1 || H < 1 || T < 0 || N < 1 || d_v < 4 || W < 1 || R < 1) return false;
  const int C = backward_cols(d_v);
  if (!C) return false;
  auto up16 = [](size_t x) { return (x + 15) & ~size_t(15); };
  const size_t lim = size_t(1) << 62;
  const double approx = double(B) * H * (double(T) * (d_v / C) * (2.0 * W + R) * 4 + double(N) * 4 +
                                         double(T) * bwd_flag_words(W, R) * 4 +
                                         double(T) * (W + R) * 4);
  if (approx > double(lim)) return false;
  const size_t bh = size_t(B) * size_t(H);
  ws->part = up16(bh * size_t(T) * size_t(d_v / C) * size_t(2 * W + R) * 4);
  ws->wts = up16(bh * size_t(T) * size_t(W + R) * 4);
  ws->flags = up16(bh * size_t(T) * size_t(bwd_flag_words(W, R)) * 4);
  ws->last = (flags & SDM_BWD_FINAL_ZERO) ? up16(bh * size_t(N) * 4) : 0;
  ws->total = ws->part + ws->wts + ws->flags + ws->last;
  return true;
}

int grid_for(size_t work, int per_block) {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return -1;
  size_t blocks = (work + per_block - 1) / per_block;
  const size_t cap = size_t(sms) * 8;
  return int(blocks < cap ? (blocks < 1 ? 1 : blocks) : cap);
}

}  // namespace
}  // namespace sdm

using namespace sdm;

extern "C" {

size_t sdm_scan_backward_workspace_size(int B, int H, int T, int d_v, int W, int R) {
  if (T < 1) return 0;
  BwdWorkspace ws;
  return backward_workspace(B, H, T, 1, d_v, W, R, 0u, &ws) ? ws.total : 0;
}

size_t sdm_scan_backward_workspace_size_ex(int B, int H, int T, long long N, int d_v, int W, int R,
                                           unsigned flags) {
  if (flags & ~unsigned(SDM_BWD_FINAL_ZERO | SDM_BWD_DM0_ONLY)) return 0;
  BwdWorkspace ws;
  return backward_workspace(B, H, T, N, d_v, W, R, flags, &ws) ? ws.total : 0;
}

int sdm_scan_forward_train(float* M, const int32_t* idx_w, const float* sc_w,
                           const int32_t* idx_r, const float* sc_r, const void* v, int v_dt,
                           const float* alpha, const float* beta, int B, int H, int T,
                           long long N, int d_v, int W, int R, float* o, float* w_prev,
                           float* r_rows, void* workspace, size_t workspace_bytes, int* dev_err,
                           void* stream) {
  int st = check_scan_args(M, idx_w, sc_w, idx_r, sc_r, v, v_dt, alpha, beta, B, H, T, N, d_v, W,
                           R, o);
  if (st != SDM_OK) return st;
  if (T == 0) return SDM_OK;
  if (!aligned16(w_prev) || !aligned16(r_rows) || !aligned16(workspace)) return SDM_EALIGN;
  if (workspace_bytes < sdm_scan_workspace_size(B, H, T, d_v, W, R)) return SDM_ENOSPACE;
  if (dev_err && (reinterpret_cast<uintptr_t>(dev_err) & 3u)) return SDM_EALIGN;
  ScanShape shape;
  st = choose_scan_shape(B * H, d_v, W, R, 0, 0, &shape);
  if (st != SDM_OK) return st;
  return launch_scan(M, idx_w, sc_w, idx_r, sc_r, v, v_dt, alpha, beta, whole_sequences(B * H, T),
                     N, d_v, W, R, o, workspace, dev_err, shape, nullptr, nullptr,
                     as_stream(stream), w_prev, r_rows);
}

int sdm_scan_backward(const int32_t* idx_w, const float* sc_w, const int32_t* idx_r,
                      const float* sc_r, const void* v, int v_dt, const float* alpha,
                      const float* beta, const float* w_prev, const float* r_rows,
                      const float* dO, int B, int H, int T, long long N, int d_v, int W, int R,
                      float* G, float* dv, float* dalpha, float* dbeta, float* dsc_w,
                      float* dsc_r, float* dM0, void* workspace, size_t workspace_bytes,
                      void* stream) {
  return sdm_scan_backward_ex(idx_w, sc_w, idx_r, sc_r, v, v_dt, alpha, beta, w_prev, r_rows, dO, B,
                              H, T, N, d_v, W, R, G, dv, dalpha, dbeta, dsc_w, dsc_r, dM0, 0u,
                              workspace, workspace_bytes, stream);
}

int sdm_scan_backward_ex(const int32_t* idx_w, const float* sc_w, const int32_t* idx_r,
                         const float* sc_r, const void* v, int v_dt, const float* alpha,
                         const float* beta, const float* w_prev, const float* r_rows,
                         const float* dO, int B, int H, int T, long long N, int d_v, int W, int R,
                         float* G, float* dv, float* dalpha, float* dbeta, float* dsc_w,
                         float* dsc_r, float* dM0, unsigned flags, void* workspace,
                         size_t workspace_bytes, void* stream) {
  if (flags & ~unsigned(SDM_BWD_FINAL_ZERO | SDM_BWD_DM0_ONLY)) return SDM_EINVAL;
  const bool zero_final = (flags & SDM_BWD_FINAL_ZERO) != 0;
  const bool dm0_only = (flags & SDM_BWD_DM0_ONLY) != 0;
  if (dm0_only && !dM0) return SDM_EINVAL;
  int st = check_scan_args(G, idx_w, sc_w, idx_r, sc_r, v, v_dt, alpha, beta, B, H, T, N, d_v, W,
                           R, dv);
  if (st != SDM_OK) return st;
  const int C = backward_cols(d_v);
  if (!C) return SDM_EUNSUPPORTED;
  cudaStream_t s = as_stream(stream);
  const size_t per_batch4 = size_t(H) * size_t(N) * d_v / 4;
  if (dM0 && !aligned16(dM0)) return SDM_EALIGN;
  BwdWorkspace ws;
  if (!backward_workspace(B, H, T, N, d_v, W, R, flags, &ws)) return SDM_EUNSUPPORTED;
  if ((T > 0 || zero_final) && !aligned16(workspace)) return SDM_EALIGN;
  if ((T > 0 || zero_final) && workspace_bytes < ws.total) return SDM_ENOSPACE;
  unsigned char* wsb = static_cast<unsigned char*>(workspace);
  float* wts = reinterpret_cast<float*>(wsb + ws.part);
  uint32_t* fl = reinterpret_cast<uint32_t*>(wsb + ws.part + ws.wts);
  int32_t* last =
      zero_final ? reinterpret_cast<int32_t*>(wsb + ws.part + ws.wts + ws.flags) : nullptr;
  const int NW = (W + R + 31) / 32, NS = (W + 31) / 32;
  const long long tokens = (long long)B * H * T;
  if (zero_final) {
    if (launch_fill_words(last, -1, size_t(B) * size_t(H) * size_t(N), s) != SDM_OK)
      return SDM_ECUDA;
    if (tokens > 0) {
      const long long tb = (tokens + 7) / 8;
      if (tb > 0x7FFFFFFFLL) return SDM_EUNSUPPORTED;
      last_read_kernel<<<unsigned(tb), 256, 0, s>>>(idx_r, T, R, N, tokens, last);
      if (last_launch_status() != SDM_OK) return SDM_ECUDA;
    }
  }
  if (tokens > 0) {
    int l = 5;
    while ((1 << l) < 2 * R) ++l;
    const int warps = int(min(size_t(8), size_t(48 * 1024) / (size_t(4) << l)));
    const long long fb = (tokens + warps - 1) / warps;
    if (fb > 0x7FFFFFFFLL || warps < 1) return SDM_EUNSUPPORTED;
    bwd_flags_kernel<<<unsigned(fb), warps * 32, size_t(warps) * (size_t(4) << l), s>>>(
        idx_w, idx_r, T, W, R, N, tokens, last, NW, NS, bwd_flag_words(W, R), l, fl);
    if (last_launch_status() != SDM_OK) return SDM_ECUDA;
  }
  if (T > 0) {
    if (!aligned16(w_prev) || !aligned16(r_rows) || !aligned16(dO) || !aligned16(dalpha) ||
        !aligned16(dbeta) || !aligned16(dsc_w) || !aligned16(dsc_r))
      return SDM_EALIGN;
    const long long wb = (tokens + 7) / 8;
    if (wb > 0x7FFFFFFFLL) return SDM_EUNSUPPORTED;
    bwd_weights_kernel<<<unsigned(wb), 256, 0, s>>>(sc_w, sc_r, W, R, tokens, wts);
    if (last_launch_status() != SDM_OK) return SDM_ECUDA;
    BwdArgs a;
    a.idx_w = idx_w;
    a.sc_w = sc_w;
    a.idx_r = idx_r;
    a.sc_r = sc_r;
    a.v = v;
    a.v_bf16 = v_dt == SDM_BF16;
    a.alpha = alpha;
    a.beta = beta;
    a.w_prev = w_prev;
    a.r_rows = r_rows;
    a.dO = dO;
    a.G = G;
    a.dv = dv;
    a.part = reinterpret_cast<float*>(wsb);
    a.wts = wts;
    a.flags = fl;
    a.NW = NW;
    a.NS = NS;
    a.NF = bwd_flag_words(W, R);
    a.vec16 = W % 4 == 0 && R % 4 == 0 && aligned16(idx_w) && aligned16(idx_r);
    a.zero_final = zero_final;
    a.T = T;
    a.N = N;
    a.d_v = d_v;
    a.W = W;
    a.R = R;
    const int smem = int(backward_smem_bytes(C, W, R, a.NF));
    const void* fn = C == 32   ? reinterpret_cast<const void*>(&scan_backward_kernel<32>)
                     : C == 16 ? reinterpret_cast<const void*>(&scan_backward_kernel<16>)
                     : C == 8  ? reinterpret_cast<const void*>(&scan_backward_kernel<8>)
                               : reinterpret_cast<const void*>(&scan_backward_kernel<4>);
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
      return SDM_ECUDA;
    void* args[] = {&a};
    if (cudaLaunchKernel(fn, dim3(unsigned(B * H * (d_v / C))), dim3(kBwdThreads), args,
                         size_t(smem), s) != cudaSuccess)
      return SDM_ECUDA;
    // finish: one warp per (b, h, t)
    const long long items = tokens;
    const int fsmem = 4 * 2 * (W + R) * 4;
    if (cudaFuncSetAttribute(reinterpret_cast<const void*>(&backward_finish_kernel),
                             cudaFuncAttributeMaxDynamicSharedMemorySize, fsmem) != cudaSuccess)
      return SDM_ECUDA;
    backward_finish_kernel<<<unsigned((items + 3) / 4), 128, fsmem, s>>>(
        wts, beta, a.part, d_v / C, W, R, items, dalpha, dbeta, dsc_w, dsc_r);
    if (last_launch_status() != SDM_OK) return SDM_ECUDA;
  }
  if (zero_final) {
    const long long rows = (long long)H * N;
    const int blocks = grid_for(size_t(B <= 32 ? (rows + 31) / 32 : rows), 8);
    if (blocks < 1) return SDM_ECUDA;
    if (B <= 32)
      reduce_batch_zero_kernel<<<blocks, 256, 0, s>>>(reinterpret_cast<float4*>(G),
                                                       reinterpret_cast<float4*>(dM0), last, B, rows,
                                                       d_v / 4, !dm0_only);
    else
      reduce_batch_zero_wide_kernel<<<blocks, 256, 0, s>>>(reinterpret_cast<float4*>(G),
                                                            reinterpret_cast<float4*>(dM0), last, B,
                                                            rows, d_v / 4, !dm0_only);
    return last_launch_status();
  }
  if (dM0) {
    const int blocks = grid_for(per_batch4, 256);
    if (blocks < 1) return SDM_ECUDA;
    reduce_batch_kernel<<<blocks, 256, 0, s>>>(reinterpret_cast<const float4*>(G),
                                                reinterpret_cast<float4*>(dM0), B, per_batch4);
    return last_launch_status();
  }
  return SDM_OK;
}

int sdm_select_backward(const int32_t* idx, const float* dsc, int B, int H, int T, int S, int K,
                        float* dhalves, void* stream) {
  if (B < 1 || H < 1 || T < 0 || S < 1 || K < 1 || (long long)K > (long long)S * S)
    return SDM_EINVAL;
  if (S > SDM_MAX_S || K > SDM_MAX_K) return SDM_EUNSUPPORTED;
  const long long items = (long long)B * H * T;
  if (items == 0) return SDM_OK;
  if (!aligned16(idx) || !aligned16(dsc) || !aligned16(dhalves)) return SDM_EALIGN;
  select_backward_kernel<<<unsigned((items + 3) / 4), 128, 0, as_stream(stream)>>>(idx, dsc, items,
                                                                                  S, K, dhalves);
  return last_launch_status();
}

}  // extern "C"
