// Synthetic input generator (not part of the method): the device twin of the host
// generator that feeds the CPU reference, reproducing its draws bit for bit so that
// large workloads can be drawn straight into HBM.
//
//   Philox4x32-10 (Salmon, Moraes, Dror, Shaw, SC'11): key = (seed lo, seed hi),
//   counter = (e lo, e hi, field, 0), e = row-major element index in the full logical
//   tensor.  Uniform u1 = ((x0 >> 8) + 1) 2^-24 in (0, 1]; angle = 2 pi (x1 >> 8) / 2^24;
//   normal = sqrt(-2 ln u1) cos(angle) (Box-Muller), where ln, cos, sin and exp are
//   fixed series evaluated with explicitly rounded fp32 operations (__fadd_rn and
//   friends never contract into FMAs), so every IEEE machine produces the same bits:
//     ln u  = e ln2 + 2 z (1 + z^2/3 + z^4/5 + z^6/7 + z^8/9), z = (f-1)/(f+1),
//             u = f 2^e with f in [sqrt(1/2), sqrt(2));
//     sin/cos on [0, pi/2): Taylor series to degree 13 / 14 after an exact quadrant
//             split of the 24-bit angle;
//     exp x = 2^n p(r), n = floor(x log2 e + 1/2), r = (x - n ln2_hi) - n ln2_lo
//             (ln2 split into a high part with trailing zero bits, so n ln2_hi is exact,
//             and the rest: the argument reduction of Cody and Waite, "Software Manual
//             for the Elementary Functions", 1980), p = Taylor series to degree 8.
#include "sdm_internal.cuh"

namespace sdm {
namespace {

enum { kFieldKp = 0, kFieldQp = 1, kFieldV = 2, kFieldAlpha = 3, kFieldBeta = 4, kFieldM0 = 5 };

__device__ __forceinline__ float bitsf(uint32_t b) { return __uint_as_float(b); }

__device__ __forceinline__ void philox(uint32_t c[4], uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    if (r) {
      k0 += 0x9E3779B9u;
      k1 += 0xBB67AE85u;
    }
    const uint32_t lo0 = 0xD2511F53u * c[0], hi0 = __umulhi(0xD2511F53u, c[0]);
    const uint32_t lo1 = 0xCD9E8D57u * c[2], hi1 = __umulhi(0xCD9E8D57u, c[2]);
    const uint32_t n0 = hi1 ^ c[1] ^ k0, n2 = hi0 ^ c[3] ^ k1;
    c[0] = n0;
    c[1] = lo1;
    c[2] = n2;
    c[3] = lo0;
  }
}

__device__ __forceinline__ void draw(unsigned long long seed, int field, unsigned long long e,
                                     uint32_t& x0, uint32_t& x1) {
  uint32_t c[4] = {uint32_t(e), uint32_t(e >> 32), uint32_t(field), 0u};
  philox(c, uint32_t(seed), uint32_t(seed >> 32));
  x0 = c[0];
  x1 = c[1];
}

__device__ __forceinline__ float uniform_open(uint32_t x0) {
  return __fmul_rn(__fadd_rn(float(x0 >> 8), 1.0f), bitsf(0x33800000u));  // * 2^-24
}

__device__ float fixed_ln(float u) {
  const uint32_t bits = __float_as_uint(u);
  int e = int(bits >> 23) - 127;
  float f = bitsf((bits & 0x7FFFFFu) | 0x3F800000u);
  if (f > bitsf(0x3FB504F3u)) {  // sqrt(2)
    f = __fmul_rn(f, 0.5f);
    e += 1;
  }
  const float z = __fdiv_rn(__fsub_rn(f, 1.0f), __fadd_rn(f, 1.0f));
  const float z2 = __fmul_rn(z, z);
  float p = bitsf(0x3DE38E39u);                          // 1/9
  p = __fadd_rn(__fmul_rn(p, z2), bitsf(0x3E124925u));   // 1/7
  p = __fadd_rn(__fmul_rn(p, z2), bitsf(0x3E4CCCCDu));   // 1/5
  p = __fadd_rn(__fmul_rn(p, z2), bitsf(0x3EAAAAABu));   // 1/3
  p = __fadd_rn(__fmul_rn(p, z2), 1.0f);
  const float t = __fmul_rn(z, p);
  return __fadd_rn(__fmul_rn(float(e), bitsf(0x3F317218u)), __fadd_rn(t, t));
}

__device__ float fixed_cos_turn(uint32_t k24) {
  const uint32_t quad = k24 >> 22;
  const float phi = __fmul_rn(float(k24 & 0x3FFFFFu), bitsf(0x34C90FDBu));  // (pi/2) 2^-22
  const float p2 = __fmul_rn(phi, phi);
  float s = bitsf(0x2F309231u);                          //  1/13!
  s = __fadd_rn(__fmul_rn(s, p2), bitsf(0xB2D7322Bu));   // -1/11!
  s = __fadd_rn(__fmul_rn(s, p2), bitsf(0x3638EF1Du));   //  1/9!
  s = __fadd_rn(__fmul_rn(s, p2), bitsf(0xB9500D01u));   // -1/7!
  s = __fadd_rn(__fmul_rn(s, p2), bitsf(0x3C088889u));   //  1/5!
  s = __fadd_rn(__fmul_rn(s, p2), bitsf(0xBE2AAAABu));   // -1/3!
  s = __fmul_rn(phi, __fadd_rn(__fmul_rn(s, p2), 1.0f));
  float c = bitsf(0xAD49CBA5u);                          // -1/14!
  c = __fadd_rn(__fmul_rn(c, p2), bitsf(0x310F76C7u));   //  1/12!
  c = __fadd_rn(__fmul_rn(c, p2), bitsf(0xB493F27Eu));   // -1/10!
  c = __fadd_rn(__fmul_rn(c, p2), bitsf(0x37D00D01u));   //  1/8!
  c = __fadd_rn(__fmul_rn(c, p2), bitsf(0xBAB60B61u));   // -1/6!
  c = __fadd_rn(__fmul_rn(c, p2), bitsf(0x3D2AAAABu));   //  1/4!
  c = __fadd_rn(__fmul_rn(c, p2), bitsf(0xBF000000u));   // -1/2!
  c = __fadd_rn(__fmul_rn(c, p2), 1.0f);
  return quad == 0 ? c : (quad == 1 ? -s : (quad == 2 ? -c : s));
}

__device__ float fixed_exp(float x) {
  const float n = floorf(__fadd_rn(__fmul_rn(x, bitsf(0x3FB8AA3Bu)), 0.5f));  // log2(e)
  const float r = __fsub_rn(__fsub_rn(x, __fmul_rn(n, bitsf(0x3F317200u))), __fmul_rn(n, bitsf(0x35BFBE8Eu)));
  float p = bitsf(0x37D00D01u);                          // 1/8!
  p = __fadd_rn(__fmul_rn(p, r), bitsf(0x39500D01u));    // 1/7!
  p = __fadd_rn(__fmul_rn(p, r), bitsf(0x3AB60B61u));    // 1/6!
  p = __fadd_rn(__fmul_rn(p, r), bitsf(0x3C088889u));    // 1/5!
  p = __fadd_rn(__fmul_rn(p, r), bitsf(0x3D2AAAABu));    // 1/4!
  p = __fadd_rn(__fmul_rn(p, r), bitsf(0x3E2AAAABu));    // 1/3!
  p = __fadd_rn(__fmul_rn(p, r), bitsf(0x3F000000u));    // 1/2!
  p = __fadd_rn(__fmul_rn(__fadd_rn(__fmul_rn(p, r), 1.0f), r), 1.0f);
  const float scale = __uint_as_float(uint32_t(int(n) + 127) << 23);
  return __fmul_rn(p, scale);
}

__device__ __forceinline__ float normal_at(unsigned long long seed, int field,
                                           unsigned long long e) {
  uint32_t x0, x1;
  draw(seed, field, e, x0, x1);
  const float r = __fsqrt_rn(__fmul_rn(-2.0f, fixed_ln(uniform_open(x0))));
  return __fmul_rn(r, fixed_cos_turn(x1 >> 8));
}

__device__ __forceinline__ float uniform_at(unsigned long long seed, int field,
                                            unsigned long long e) {
  uint32_t x0, x1;
  draw(seed, field, e, x0, x1);
  return uniform_open(x0);
}

__device__ __forceinline__ uint16_t bf16_rne(float x) {
  const uint32_t u = __float_as_uint(x);
  return uint16_t((u + 0x7FFFu + ((u >> 16) & 1u)) >> 16);
}

__device__ __forceinline__ void store(void* out, size_t i, float x, bool bf16) {
  if (bf16)
    static_cast<uint16_t*>(out)[i] = bf16_rne(x);
  else
    static_cast<float*>(out)[i] = x;
}

struct GenBox {
  unsigned long long seed;
  int B, H, T, b_off, t_off;
  long long T_total;
  int S, d_v;
  bool bf16;
};

// global (b, h, t) row index of box-local (b, h, t)
__device__ __forceinline__ unsigned long long bht_global(const GenBox& g, size_t b, size_t h,
                                                          size_t t) {
  return ((unsigned long long)(b + g.b_off) * g.H + h) * (unsigned long long)g.T_total +
         (unsigned long long)(t + g.t_off);
}

__global__ void gen_halves_kernel(GenBox g, int field, const float* __restrict__ bias, void* out) {
  const size_t total = size_t(g.B) * g.H * g.T * 2 * g.S;
  const size_t stride = size_t(gridDim.x) * blockDim.x;
  for (size_t i = size_t(blockIdx.x) * blockDim.x + threadIdx.x; i < total; i += stride) {
    const size_t j = i % g.S;
    size_t r = i / g.S;
    const size_t half = r % 2;
    r /= 2;
    const size_t t = r % g.T;
    r /= g.T;
    const size_t h = r % g.H, b = r / g.H;
    const unsigned long long e = (bht_global(g, b, h, t) * 2 + half) * g.S + j;
    float x = normal_at(g.seed, field, e);
    if (bias) x = __fadd_rn(x, bias[j]);
    store(out, i, x, g.bf16);
  }
}

__global__ void gen_v_kernel(GenBox g, void* out) {
  const size_t total = size_t(g.B) * g.H * g.T * g.d_v;
  const size_t stride = size_t(gridDim.x) * blockDim.x;
  for (size_t i = size_t(blockIdx.x) * blockDim.x + threadIdx.x; i < total; i += stride) {
    const size_t c = i % g.d_v;
    size_t r = i / g.d_v;
    const size_t t = r % g.T;
    r /= g.T;
    const size_t h = r % g.H, b = r / g.H;
    const unsigned long long e = bht_global(g, b, h, t) * g.d_v + c;
    store(out, i, normal_at(g.seed, kFieldV, e), g.bf16);
  }
}

__global__ void gen_gates_kernel(GenBox g, float alpha_lo, int beta_kind, float* alpha,
                                 float* beta) {
  const size_t total = size_t(g.B) * g.H * g.T;
  const size_t stride = size_t(gridDim.x) * blockDim.x;
  const float span = __fsub_rn(1.0f, alpha_lo);
  for (size_t i = size_t(blockIdx.x) * blockDim.x + threadIdx.x; i < total; i += stride) {
    const size_t t = i % g.T;
    const size_t r = i / g.T;
    const size_t h = r % g.H, b = r / g.H;
    const unsigned long long e = bht_global(g, b, h, t);
    if (alpha) alpha[i] = __fadd_rn(alpha_lo, __fmul_rn(span, uniform_at(g.seed, kFieldAlpha, e)));
    if (beta) {
      if (beta_kind == 0) {
        beta[i] = uniform_at(g.seed, kFieldBeta, e);
      } else {
        const float z = normal_at(g.seed, kFieldBeta, e);
        beta[i] = __fdiv_rn(1.0f, __fadd_rn(1.0f, fixed_exp(-z)));
      }
    }
  }
}

__global__ void gen_m0_kernel(unsigned long long seed, size_t total, float scale, float* M0) {
  const size_t stride = size_t(gridDim.x) * blockDim.x;
  for (size_t i = size_t(blockIdx.x) * blockDim.x + threadIdx.x; i < total; i += stride)
    M0[i] = __fmul_rn(scale, normal_at(seed, kFieldM0, i));
}

unsigned grid_for(size_t total) {
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess)
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const size_t want = (total + 255) / 256;
  const size_t cap = size_t(sms) * 16;
  return unsigned(want < cap ? (want ? want : 1) : cap);
}

}  // namespace

int launch_gen_inputs(unsigned long long seed, int B, int H, int T, int b_off, int t_off,
                      long long T_total, int S, int d_v, int in_dt, float alpha_lo,
                      int beta_kind, const float* half_bias, void* kp, void* qp, void* v,
                      float* alpha, float* beta, cudaStream_t s) {
  GenBox g{seed, B, H, T, b_off, t_off, T_total, S, d_v, in_dt == SDM_BF16};
  const size_t bht = size_t(B) * H * T;
  if (bht == 0) return SDM_OK;
  if (kp) gen_halves_kernel<<<grid_for(bht * 2 * S), 256, 0, s>>>(g, kFieldKp, half_bias, kp);
  if (qp) gen_halves_kernel<<<grid_for(bht * 2 * S), 256, 0, s>>>(g, kFieldQp, half_bias, qp);
  if (v) gen_v_kernel<<<grid_for(bht * d_v), 256, 0, s>>>(g, v);
  if (alpha || beta) gen_gates_kernel<<<grid_for(bht), 256, 0, s>>>(g, alpha_lo, beta_kind, alpha, beta);
  return last_launch_status();
}

int launch_gen_M0(unsigned long long seed, int H, long long N, int d_v, float scale, float* M0,
                  cudaStream_t s) {
  const size_t total = size_t(H) * size_t(N) * size_t(d_v);
  if (total == 0) return SDM_OK;
  gen_m0_kernel<<<grid_for(total), 256, 0, s>>>(seed, total, scale, M0);
  return last_launch_status();
}

}  // namespace sdm
