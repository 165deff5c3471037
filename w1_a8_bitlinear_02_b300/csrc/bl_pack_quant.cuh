// Weight ternarisation + packing, and activation quantisation kernels.
//
// Weights: absmean ternarisation, one fp32 scale per tensor ("20亿参数仅0.4GB…
// 「原生1.58bit」大模型", blog.csdn.net/soaring_casia, section 2 "BitLinear层",
// item 1).  Activations: per-token absmax to int8 (same section, item 2).
// The fused variant applies the subln RMSNorm first (item 3).
#pragma once

#include <cuda_bf16.h>
#include <cstdint>

#include "bl_ptx.cuh"

namespace bl {

__device__ __forceinline__ float to_f32(float v) { return v; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }

// ------------------------------------------------------------------ pack
// Row sums of |W| in fp64, each row added sequentially over k.  A block
// owns 256 rows; 32-column slabs are staged through shared memory so the
// global reads are coalesced while every row keeps its k order.
template <typename WT>
__global__ void __launch_bounds__(256) pack_rowsum_kernel(const WT *__restrict__ W, int64_t N,
                                                          int64_t K, double *__restrict__ rowsum) {
  __shared__ float tile[256][33];
  const int64_t n0 = static_cast<int64_t>(blockIdx.x) * 256;
  const int t = threadIdx.x;
  double acc = 0.0;
  for (int64_t k0 = 0; k0 < K; k0 += 32) {
#pragma unroll 4
    for (int i = 0; i < 32; ++i) {
      const int r = (t >> 5) + 8 * i;
      const int c = t & 31;
      const int64_t n = n0 + r, k = k0 + c;
      tile[r][c] = (n < N && k < K) ? to_f32(W[n * K + k]) : 0.0f;
    }
    __syncthreads();
    const int kmax = static_cast<int>(K - k0 < 32 ? K - k0 : 32);
    for (int c = 0; c < kmax; ++c) acc += fabs(static_cast<double>(tile[t][c]));
    __syncthreads();
  }
  if (n0 + t < N) rowsum[n0 + t] = acc;
}

// gamma = fl32( fl32(S / (N*K)) + 1e-5f ), S = row sums added in row order.
__global__ void pack_gamma_kernel(const double *__restrict__ rowsum, int64_t N, int64_t K,
                                  float *__restrict__ gamma) {
  if (threadIdx.x != 0 || blockIdx.x != 0) return;
  double S = 0.0;
  for (int64_t n = 0; n < N; ++n) S = __dadd_rn(S, rowsum[n]);
  const float mean = __double2float_rn(__ddiv_rn(S, static_cast<double>(N) * static_cast<double>(K)));
  *gamma = __fadd_rn(mean, 1e-5f);
}

// Grouped weights: gamma_g = fl32( fl32(S_g / (G*K)) + 1e-5f ) for each group
// of G consecutive rows, S_g its row sums added in row order (one thread per
// group, so the order is the same as the per-tensor scale's).
__global__ void pack_gamma_groups_kernel(const double *__restrict__ rowsum, int64_t groups, int64_t G,
                                         int64_t K, float *__restrict__ gamma) {
  const int64_t g = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (g >= groups) return;
  double S = 0.0;
  for (int64_t n = g * G; n < (g + 1) * G; ++n) S = __dadd_rn(S, rowsum[n]);
  const float mean = __double2float_rn(__ddiv_rn(S, static_cast<double>(G) * static_cast<double>(K)));
  gamma[g] = __fadd_rn(mean, 1e-5f);
}

// One thread per 32-bit packed word (16 weights).  Code = clip(rint(W/gamma))+1;
// weight k = 16w + 4i + j goes to bit 8j + 2i; k >= K gets code 1.  Row n
// takes gamma[n >> glog2]; glog2 < 0: the one per-tensor scale gamma[0].
template <typename WT>
__global__ void __launch_bounds__(256) pack_codes_kernel(const WT *__restrict__ W, int64_t N,
                                                         int64_t K, int64_t words_per_row,
                                                         const float *__restrict__ gamma, int glog2,
                                                         uint32_t *__restrict__ packed) {
  const int64_t id = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (id >= N * words_per_row) return;
  const int64_t n = id / words_per_row;
  const int64_t w = id - n * words_per_row;
  const float g = gamma[glog2 < 0 ? 0 : (n >> glog2)];
  const WT *row = W + n * K;
  uint32_t word = 0;
#pragma unroll
  for (int t = 0; t < 16; ++t) {
    const int64_t k = 16 * w + t;
    uint32_t code = 1u;
    if (k < K) {
      float q = rintf(__fdiv_rn(to_f32(row[k]), g));
      q = fminf(fmaxf(q, -1.0f), 1.0f);
      code = static_cast<uint32_t>(static_cast<int>(q) + 1);
    }
    word |= code << (8 * (t & 3) + 2 * (t >> 2));
  }
  packed[id] = word;
}

// ------------------------------------------------------------------ quant
// Block-wide reductions over the first `nthreads` threads of a block
// (a multiple of 32), using named barrier `bar_id`.
__device__ __forceinline__ void named_bar(int bar_id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(bar_id), "r"(nthreads) : "memory");
}

// Barrier over the first `nthreads` threads that also ORs a predicate.
__device__ __forceinline__ bool named_bar_or(int bar_id, int nthreads, bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "barrier.cta.red.or.pred q, %2, %3, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(v)), "r"(bar_id), "r"(nthreads)
      : "memory");
  return r != 0u;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Max over a warp of non-negative floats: their bit patterns order like
// unsigned integers, so one redux instruction does it.
__device__ __forceinline__ float warp_max_nonneg(float v) {
  return __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(v)));
}

__device__ __forceinline__ double warp_sum_f64(double v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// xq = clip(rint(fl32(v * s)), -128, 127)
__device__ __forceinline__ int quant_one(float v, float s) {
  float r = rintf(__fmul_rn(v, s));
  r = fminf(fmaxf(r, -128.0f), 127.0f);
  return static_cast<int>(r);
}

// Activation applied before quantisation: 0 none, 1 squared ReLU
// fl32(max(x, 0)^2) (the FFN activation feeding the down projection).
constexpr int kActNone = 0;
constexpr int kActRelu2 = 1;
__device__ __forceinline__ float relu2f(float v) {
  const float r = fmaxf(v, 0.0f);
  return __fmul_rn(r, r);
}

// Where a forward writes y[i] = v: fp32 or bf16 (one round to nearest even),
// adding first, in fp32, a residual of the output's dtype when one is given
// (it may be y itself: each element is read and then written by one thread).
struct OutSpec {
  void *y;                      // [M, N] fp32 or bf16
  const void *res;              // [M, N] of the same dtype, or null
  int bf16;
  const float *gvec = nullptr;  // grouped weights: one scale per 2^glog2 output rows, else null
  int glog2 = 0;
};

// Grouped weights: the output scale of token m at row n is fl32(gamma_g / s_m)
// with g row n's group (per-tensor weights use c_m = fl32(gamma / s_m),
// computed once per token).
__device__ __forceinline__ float group_scale(const OutSpec &o, int64_t n, float s_m) {
  return __fdiv_rn(__ldg(o.gvec + (n >> o.glog2)), s_m);
}
__device__ __forceinline__ void put_y(const OutSpec &o, int64_t i, float v) {
  if (o.res != nullptr)
    v = __fadd_rn(v, o.bf16 ? __bfloat162float(static_cast<const __nv_bfloat16 *>(o.res)[i])
                            : static_cast<const float *>(o.res)[i]);
  if (o.bf16)
    static_cast<__nv_bfloat16 *>(o.y)[i] = __float2bfloat16_rn(v);
  else
    static_cast<float *>(o.y)[i] = v;
}

__device__ __forceinline__ float act_scale(float amax) {
  return __fdiv_rn(127.0f, fmaxf(amax, 1e-5f));
}

// Zero row m of an int32 [M, zn] accumulator and (block 0) ncnt tickets: the
// split-K contraction that follows on the stream adds into them.
__device__ __forceinline__ void zero_fill(int64_t m, int32_t *zrows, int64_t zn, unsigned *zcnt,
                                          int ncnt) {
  if (zrows != nullptr)
    for (int64_t k = threadIdx.x; k < zn; k += blockDim.x) zrows[m * zn + k] = 0;
  if (zcnt != nullptr && m == 0)
    for (int i = threadIdx.x; i < ncnt; i += blockDim.x) zcnt[i] = 0u;
}

// 8 consecutive activations as floats (16- or 32-byte vector loads).
__device__ __forceinline__ void load8(const float *p, float (&v)[8]) {
  const float4 a = __ldg(reinterpret_cast<const float4 *>(p));
  const float4 b = __ldg(reinterpret_cast<const float4 *>(p) + 1);
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
  v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}
__device__ __forceinline__ void load8(const __nv_bfloat16 *p, float (&v)[8]) {
  const uint4 u = __ldg(reinterpret_cast<const uint4 *>(p));
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    v[2 * j] = __uint_as_float(w[j] << 16);
    v[2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
  }
}

__device__ __forceinline__ bool al16(const void *p) {
  return (reinterpret_cast<uintptr_t>(p) & 15u) == 0u;
}

// Kahan step: (s, c) += y  (compensated fp32 sum of squares)
__device__ __forceinline__ void kahan_add(float &s, float &c, float y) {
  const float yy = __fsub_rn(y, c);
  const float t = __fadd_rn(s, yy);
  c = __fsub_rn(__fsub_rn(t, s), yy);
  s = t;
}

// One block (256 threads) per token row.
//   OUT_BF16 = false: xq int8 [M, K] dense.
//   OUT_BF16 = true : integer codes as bf16 [M, ld] (exact), zero for k in [K, ld);
//                     the tensor-core path reads this layout.
//   NORM: fused subln RMSNorm (gain g may be NULL).
//   act: kActRelu2 squares the positive part of x first (not with NORM).
// Rows are read in 8-element vectors (two passes: max, then codes; the second
// pass hits L1) when K and the pointers allow, else element by element.
template <typename XT, bool OUT_BF16, bool NORM>
__global__ void __launch_bounds__(256) quant_act_kernel(const XT *__restrict__ x, int64_t K,
                                                        int64_t ld, const float *__restrict__ g,
                                                        float eps, int8_t *__restrict__ xq,
                                                        __nv_bfloat16 *__restrict__ xb,
                                                        float *__restrict__ scale,
                                                        int32_t *__restrict__ zrows, int64_t zn,
                                                        unsigned *__restrict__ zcnt, int ncnt, int act) {
  __shared__ float red_f[8];
  __shared__ double red_d[8];
  pdl_wait_primary();
  pdl_launch_dependents();
  const int64_t m = blockIdx.x;
  const XT *xr = x + m * K;
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const bool use_g = NORM && g != nullptr;
  const bool vec = (K % 8) == 0 && al16(x) && (!use_g || al16(g)) &&
                   (OUT_BF16 ? (al16(xb) && ld % 8 == 0) : (reinterpret_cast<uintptr_t>(xq) & 7u) == 0u);
  const int64_t nvec = vec ? K / 8 : 0;

  // ---- pass 1: max |x * g| (and sum of x^2)
  float amax = 0.0f, s1 = 0.0f, c1 = 0.0f;
#pragma unroll 4
  for (int64_t c = t; c < nvec; c += 256) {
    float v[8];
    load8(xr + 8 * c, v);
    if (act == kActRelu2)
#pragma unroll
      for (int j = 0; j < 8; ++j) v[j] = relu2f(v[j]);
    float gg[8];
    if (use_g) load8(g + 8 * c, gg);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (NORM) kahan_add(s1, c1, __fmul_rn(v[j], v[j]));
      const float u = use_g ? __fmul_rn(v[j], gg[j]) : v[j];
      amax = fmaxf(amax, fabsf(u));
    }
  }
  for (int64_t k = 8 * nvec + t; k < K; k += 256) {
    float v = to_f32(xr[k]);
    if (act == kActRelu2) v = relu2f(v);
    if (NORM) kahan_add(s1, c1, __fmul_rn(v, v));
    amax = fmaxf(amax, fabsf(use_g ? __fmul_rn(v, g[k]) : v));
  }
  amax = warp_max_nonneg(amax);
  if (lane == 0) red_f[warp] = amax;
  float r_norm = 1.0f;
  if (NORM) {
    double part = static_cast<double>(s1) - static_cast<double>(c1);
    part = warp_sum_f64(part);
    if (lane == 0) red_d[warp] = part;
  }
  __syncthreads();
  amax = red_f[0];
#pragma unroll
  for (int i = 1; i < 8; ++i) amax = fmaxf(amax, red_f[i]);
  const float s = act_scale(amax);
  if (NORM) {
    double S = 0.0;
#pragma unroll
    for (int i = 0; i < 8; ++i) S += red_d[i];
    const float ms = __double2float_rn(S / static_cast<double>(K));
    const float d = __fsqrt_rn(__fadd_rn(ms, eps));
    r_norm = __fdiv_rn(1.0f, d);
  }
  if (t == 0) scale[m] = NORM ? __fdiv_rn(s, r_norm) : s;

  // ---- pass 2: codes
#pragma unroll 4
  for (int64_t c = t; c < nvec; c += 256) {
    float v[8];
    load8(xr + 8 * c, v);
    if (act == kActRelu2)
#pragma unroll
      for (int j = 0; j < 8; ++j) v[j] = relu2f(v[j]);
    float gg[8];
    if (use_g) load8(g + 8 * c, gg);
    int q[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) q[j] = quant_one(use_g ? __fmul_rn(v[j], gg[j]) : v[j], s);
    if (OUT_BF16) {
      uint32_t w[4];
#pragma unroll
      for (int j = 0; j < 4; ++j)
        w[j] = (__float_as_uint(static_cast<float>(q[2 * j])) >> 16) |
               (__float_as_uint(static_cast<float>(q[2 * j + 1])) & 0xFFFF0000u);
      *reinterpret_cast<uint4 *>(xb + m * ld + 8 * c) = make_uint4(w[0], w[1], w[2], w[3]);
    } else {
      uint32_t lo = 0, hi = 0;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        lo |= (static_cast<uint32_t>(q[j]) & 0xFFu) << (8 * j);
        hi |= (static_cast<uint32_t>(q[j + 4]) & 0xFFu) << (8 * j);
      }
      *reinterpret_cast<uint2 *>(xq + m * K + 8 * c) = make_uint2(lo, hi);
    }
  }
  for (int64_t k = 8 * nvec + t; k < K; k += 256) {
    float v = to_f32(xr[k]);
    if (act == kActRelu2) v = relu2f(v);
    const int q = quant_one(use_g ? __fmul_rn(v, g[k]) : v, s);
    if (OUT_BF16)
      xb[m * ld + k] = __float2bfloat16_rn(static_cast<float>(q));
    else
      xq[m * K + k] = static_cast<int8_t>(q);
  }
  if (OUT_BF16)
    for (int64_t k = K + t; k < ld; k += 256) xb[m * ld + k] = __float2bfloat16_rn(0.0f);
  zero_fill(m, zrows, zn, zcnt, ncnt);
}

// The same quantisation into bf16 codes (the tensor-core path's operand) in
// one pass: TPR threads per row, 256 / TPR rows per block, every value of a
// row held in registers between its absmax and its codes (K % 8 == 0,
// K <= 32 * TPR, x, xb 16-byte aligned, ld % 8 == 0; no gain vector; used
// for rows of up to 4096).  The
// results equal quant_act_kernel's (the max does not depend on the order).
template <typename XT, int TPR>
__global__ void __launch_bounds__(256) quant_rows_bf16_kernel(const XT *__restrict__ x, int64_t M, int64_t K,
                                                              int64_t ld, __nv_bfloat16 *__restrict__ xb,
                                                              float *__restrict__ scale,
                                                              int32_t *__restrict__ zrows, int64_t zn,
                                                              unsigned *__restrict__ zcnt, int ncnt, int act) {
  constexpr int RPB = 256 / TPR, NV = 4, NW = TPR / 32;
  __shared__ float red[8];
  pdl_wait_primary();
  pdl_launch_dependents();
  const int t = threadIdx.x, r = t / TPR, tr = t % TPR, lane = t & 31, warp = t >> 5;
  const int64_t m = static_cast<int64_t>(blockIdx.x) * RPB + r;
  const bool live = m < M;
  const int nvec = static_cast<int>(K / 8);
  const XT *xr = x + (live ? m : 0) * K;
  float v[NV][8];
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    const int c = tr + i * TPR;
    if (live && c < nvec) {
      load8(xr + 8 * c, v[i]);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        if (act == kActRelu2) v[i][j] = relu2f(v[i][j]);
        amax = fmaxf(amax, fabsf(v[i][j]));
      }
    }
  }
  amax = warp_max_nonneg(amax);
  if (lane == 0) red[warp] = amax;
  __syncthreads();
  float a = red[r * NW];
#pragma unroll
  for (int w = 1; w < NW; ++w) a = fmaxf(a, red[r * NW + w]);
  const float s = act_scale(a);
  if (!live) return;
  if (tr == 0) scale[m] = s;
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    const int c = tr + i * TPR;
    if (c < nvec) {
      uint32_t w[4];
#pragma unroll
      for (int j = 0; j < 4; ++j)
        w[j] = (__float_as_uint(static_cast<float>(quant_one(v[i][2 * j], s))) >> 16) |
               (__float_as_uint(static_cast<float>(quant_one(v[i][2 * j + 1], s))) & 0xFFFF0000u);
      *reinterpret_cast<uint4 *>(xb + m * ld + 8 * c) = make_uint4(w[0], w[1], w[2], w[3]);
    }
  }
  for (int64_t c = nvec + tr; c < ld / 8; c += TPR)
    *reinterpret_cast<uint4 *>(xb + m * ld + 8 * c) = make_uint4(0u, 0u, 0u, 0u);
  if (zrows != nullptr)
    for (int64_t k = tr; k < zn; k += TPR) zrows[m * zn + k] = 0;
  if (zcnt != nullptr && m == 0)
    for (int i = tr; i < ncnt; i += TPR) zcnt[i] = 0u;
}

// int8 codes [M, K] -> bf16 [M, ld] (exact), zero padded; one block per row.
__global__ void __launch_bounds__(256) codes_to_bf16_kernel(const int8_t *__restrict__ xq,
                                                            int64_t K, int64_t ld,
                                                            __nv_bfloat16 *__restrict__ xb,
                                                            int32_t *__restrict__ zrows, int64_t zn,
                                                            unsigned *__restrict__ zcnt, int ncnt) {
  pdl_wait_primary();
  pdl_launch_dependents();
  const int64_t m = blockIdx.x;
  for (int64_t k = threadIdx.x; k < ld; k += 256)
    xb[m * ld + k] = __float2bfloat16_rn(k < K ? static_cast<float>(xq[m * K + k]) : 0.0f);
  zero_fill(m, zrows, zn, zcnt, ncnt);
}

}  // namespace bl
