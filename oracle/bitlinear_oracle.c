/*
 * BitLinear W1.58A8 forward -- CPU ORACLE.
 *
 * This file is test infrastructure.  Only the test-suite, the package smoke
 * check and the benchmark's CPU-baseline leg load it.  It shares no code,
 * header, table or helper with the CUDA library: it is a plain, slow,
 * loop-by-loop restatement of the definitions, meant to be checked by eye.
 *
 * Pages this follows (cited below by short title and section):
 *   [CSDN-2B4T]  "20亿参数仅0.4GB，能耗骤降90%！微软开源全球首个2B参数「原生1.58bit」
 *                大模型" (blog.csdn.net/soaring_casia/article/details/147423941),
 *                a translation of the BitNet b1.58 2B4T technical report.
 *                Section 2 "核心创新", sub-section "BitLinear层", items 1-3.
 *   [CSDN-0.4GB] "微软AI大模型炸场：0.4GB，CPU就能跑，中国团队打造！"
 *                (blog.csdn.net/2401_84494441/article/details/147773110),
 *                section 1 "极致量化" (权重三元量化 / 激活8位量化 / 归一化方法) and
 *                section 3 "软硬协同" (GPU bullet: pack-store-load-unpack-compute).
 *   [DeepDive]   "BitNet b1.58 深度解析：微软如何用1.58位量化颠覆大模型推理范式"
 *                (chenxutan.com/d/1949.html), section 2.1 (2 bits, one unused
 *                state) and section 2.3(2) (y = (W_quant @ x_quant) * scale).
 *
 * Numeric conventions (the pages fix none of them; the readings taken are
 * the plainest ones consistent with the definitions):
 *   - fl32(.) is IEEE binary32 round-to-nearest-even; rne() is round half to
 *     even.  Every fp32 operation below is a single correctly rounded IEEE op
 *     (build with -ffp-contract=off and without fast-math).
 *   - gamma's mean |W| is summed in fp64: sequentially over k inside each row,
 *     then sequentially over the row sums.  The pages only say "absmean".
 *
 * Parity pins for every function here live in tests/test_oracle_pins.py
 * (hand-worked example, closed forms, invariants, exact-rational brute force).
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Threads used by the (integer, order-free) contraction loop.  Results do not
 * depend on it: int32 sums are exact in any order. */
static int g_threads = 1;

void bl_oracle_set_threads(int n) { g_threads = n > 0 ? n : 1; }

int bl_oracle_get_threads(void) { return g_threads; }

/* Packed row length in bytes: K rounded up to a multiple of 64 weights, two
 * bits per weight.  [DeepDive 2.1]: a ternary value is stored in a 2-bit code
 * (four states, one unused); [CSDN-0.4GB 3]: several ternary values share one
 * byte.  Rounding the row to 64 weights (16 bytes) is this library's choice. */
int64_t bl_oracle_row_bytes(int64_t K) { return ((K + 63) / 64) * 16; }

/* gamma = mean(|W|) + 1e-5  ([CSDN-2B4T 2, BitLinear item 1]: absmean weight
 * quantisation; one scale per weight tensor).
 * S is accumulated in fp64 row by row (k = 0..K-1), then the row sums are
 * added in row order.  gamma = fl32( fl32(S / (N*K)) + 1e-5f ). */
double bl_oracle_abs_sum(const float *W, int64_t N, int64_t K) {
  double S = 0.0;
  for (int64_t n = 0; n < N; ++n) {
    double row = 0.0;
    for (int64_t k = 0; k < K; ++k) row += fabs((double)W[n * K + k]);
    S += row;
  }
  return S;
}

float bl_oracle_gamma(const float *W, int64_t N, int64_t K) {
  double S = bl_oracle_abs_sum(W, N, K);
  float mean = (float)(S / ((double)N * (double)K));
  float eps = 1e-5f;
  return mean + eps;
}

/* Wq = clip( rne( fl32(W / gamma) ), -1, +1 )  ([CSDN-2B4T 2, item 1]:
 * weights mapped onto {-1, 0, +1} by the absmean scale). */
void bl_oracle_ternarize(const float *W, int64_t N, int64_t K, float gamma,
                         int8_t *q) {
  for (int64_t i = 0; i < N * K; ++i) {
    float r = W[i] / gamma;
    float t = rintf(r);
    if (t > 1.0f) t = 1.0f;
    if (t < -1.0f) t = -1.0f;
    q[i] = (int8_t)t;
  }
}

/* Packed layout (this library's choice; the pages only say "2 bits each,
 * several per byte").  Code c = q + 1 in {0, 1, 2}; 3 is never written.
 * Row n starts at byte n * row_bytes.  Weight k lives in little-endian 32-bit
 * word w = k / 16 of the row, at bit 8*j + 2*i where i = (k % 16) / 4 and
 * j = k % 4; i.e. in byte 4*w + j at bit 2*i.  Positions k >= K hold code 1
 * (weight 0). */
void bl_oracle_pack(const int8_t *q, int64_t N, int64_t K, uint8_t *packed) {
  int64_t rb = bl_oracle_row_bytes(K);
  int64_t Kp = rb * 4;
  for (int64_t n = 0; n < N; ++n) {
    uint8_t *row = packed + n * rb;
    memset(row, 0, (size_t)rb);
    for (int64_t k = 0; k < Kp; ++k) {
      int code = (k < K) ? (int)q[n * K + k] + 1 : 1;
      int64_t w = k / 16;
      int i = (int)((k % 16) / 4);
      int j = (int)(k % 4);
      row[4 * w + j] |= (uint8_t)(code << (2 * i));
    }
  }
}

/* Inverse of bl_oracle_pack: codes back to {-1,0,+1}. */
void bl_oracle_unpack(const uint8_t *packed, int64_t N, int64_t K, int8_t *q) {
  int64_t rb = bl_oracle_row_bytes(K);
  for (int64_t n = 0; n < N; ++n) {
    for (int64_t k = 0; k < K; ++k) {
      int64_t w = k / 16;
      int i = (int)((k % 16) / 4);
      int j = (int)(k % 4);
      int code = (packed[n * rb + 4 * w + j] >> (2 * i)) & 3;
      q[n * K + k] = (int8_t)(code - 1);
    }
  }
}

/* Per-token absmax int8 activation quantisation ([CSDN-2B4T 2, item 2];
 * [CSDN-0.4GB 1] 激活8位量化, "per token absmax"):
 *   amax_t = max_k |x_tk|                  (exact, order free)
 *   s_t    = fl32( 127 / max(amax_t, 1e-5) )
 *   xq_tk  = clip( rne( fl32(x_tk * s_t) ), -128, 127 )                    */
void bl_oracle_quant_act(const float *x, int64_t M, int64_t K, int8_t *xq,
                         float *s) {
  for (int64_t m = 0; m < M; ++m) {
    const float *xr = x + m * K;
    float amax = 0.0f;
    for (int64_t k = 0; k < K; ++k) {
      float a = fabsf(xr[k]);
      if (a > amax) amax = a;
    }
    float floor_ = 1e-5f;
    float d = amax > floor_ ? amax : floor_;
    float sm = 127.0f / d;
    s[m] = sm;
    for (int64_t k = 0; k < K; ++k) {
      float p = xr[k] * sm;
      float r = rintf(p);
      if (r > 127.0f) r = 127.0f;
      if (r < -128.0f) r = -128.0f;
      xq[m * K + k] = (int8_t)r;
    }
  }
}

/* Squared ReLU, the FFN activation whose output feeds the down projection
 * ([CSDN-0.4GB] section "特殊设计", bullet 激活函数: 平方ReLU instead of SwiGLU):
 *   u = fl32( r * r ),  r = x if x > 0 else 0
 * (one correctly rounded fp32 product).  Its BitLinear input is then
 * quantised per token exactly as bl_oracle_quant_act does with x. */
void bl_oracle_relu2(const float *x, int64_t n, float *u) {
  for (int64_t i = 0; i < n; ++i) {
    float r = x[i] > 0.0f ? x[i] : 0.0f;
    u[i] = r * r;
  }
}

/* Output variants of the forward's last step (this library's options; the
 * pages give the residual stream of the architecture, 0.4GB page section 2,
 * and the output precision is left open):
 *   y_out = fl32( y + r )  when a residual r is given (r widened to fp32,
 *           exact from bf16), else y;
 *   then, for a bf16 output, one round-to-nearest-even to bf16. */
static uint16_t f32_to_bf16_rne(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  /* finite inputs only (a precondition of the forward) */
  uint32_t lsb = (u >> 16) & 1u;
  u += 0x7FFFu + lsb;
  return (uint16_t)(u >> 16);
}
void bl_oracle_output(const float *y, const float *r, int64_t n, int bf16_out, float *out_f32,
                      uint16_t *out_bf16) {
  for (int64_t i = 0; i < n; ++i) {
    float v = y[i];
    if (r) v = v + r[i];
    if (bf16_out)
      out_bf16[i] = f32_to_bf16_rne(v);
    else
      out_f32[i] = v;
  }
}

/* acc[m, n] = sum_k q[n, k] * xq[m, k] in int32 ([DeepDive 2.3(2)]:
 * W_quant @ x_quant; [CSDN-0.4GB 1]: with ternary weights the product needs
 * only additions).  |acc| <= 127 * K, far inside int32. */
void bl_oracle_matmul_i32(const int8_t *q, const int8_t *xq, int64_t M,
                          int64_t N, int64_t K, int32_t *acc) {
  for (int64_t m = 0; m < M; ++m) {
#ifdef _OPENMP
#pragma omp parallel for schedule(static) num_threads(g_threads)
#endif
    for (int64_t n = 0; n < N; ++n) {
      int32_t a = 0;
      for (int64_t k = 0; k < K; ++k)
        a += (int32_t)q[n * K + k] * (int32_t)xq[m * K + k];
      acc[m * N + n] = a;
    }
  }
}

/* y[m, n] = fl32( float(acc) * c_m ),  c_m = fl32( gamma / s_m ).
 * [DeepDive 2.3(2)]: y = (W_quant @ x_quant) * scale -- one scale applied to
 * the integer product.  Here that scale is the weight scale gamma divided by
 * the token's activation scale s_m = 127/amax (which quantised x by
 * multiplication).  float(acc) is exact (|acc| < 2^24). */
void bl_oracle_rescale(const int32_t *acc, float gamma, const float *s,
                       int64_t M, int64_t N, float *y) {
  for (int64_t m = 0; m < M; ++m) {
    float c = gamma / s[m];
    for (int64_t n = 0; n < N; ++n) {
      float a = (float)acc[m * N + n];
      y[m * N + n] = a * c;
    }
  }
}

/* The whole forward from packed weights: quantise x, unpack row by row,
 * contract, rescale.  Scratch buffers are passed in by the caller:
 *   xq [M*K] int8, s [M] float, acc [M*N] int32, qrow [K] int8.            */
void bl_oracle_forward_packed(const uint8_t *packed, float gamma, int64_t N,
                              int64_t K, const float *x, int64_t M, float *y,
                              int8_t *xq, float *s, int32_t *acc) {
  bl_oracle_quant_act(x, M, K, xq, s);
  int64_t rb = bl_oracle_row_bytes(K);
#ifdef _OPENMP
#pragma omp parallel for schedule(static) num_threads(g_threads)
#endif
  for (int64_t n = 0; n < N; ++n) {
    const uint8_t *row = packed + n * rb;
    for (int64_t m = 0; m < M; ++m) {
      int32_t a = 0;
      for (int64_t k = 0; k < K; ++k) {
        int64_t w = k / 16;
        int i = (int)((k % 16) / 4);
        int j = (int)(k % 4);
        int code = (row[4 * w + j] >> (2 * i)) & 3;
        a += (int32_t)(code - 1) * (int32_t)xq[m * K + k];
      }
      acc[m * N + n] = a;
    }
  }
  bl_oracle_rescale(acc, gamma, s, M, N, y);
}

/* Scale granularity: one weight scale per group of G consecutive output rows
 * ([DeepDive 5.2]: the trainable BitLinear views W as (-1, group_size, K),
 * i.e. groups of group_size output rows, group_size = 128; [DeepDive 2.2]:
 * one scale per output row, i.e. G = 1).  The pages pair these groupings
 * with a threshold-at-mean ternariser and learnt scales; this oracle keeps
 * the absmean-round quantiser of the per-tensor case and only narrows the
 * set the mean runs over: for group g = rows [gG, gG + G),
 *   S_g     = sum over the group's rows, in row order, of the row sums of
 *             |W| (fp64, sequential over k), as for the per-tensor S;
 *   gamma_g = fl32( fl32(S_g / (G*K)) + 1e-5f );
 *   Wq[n,k] = clip( rne( fl32(W[n,k] / gamma_{n/G}) ), -1, +1 );
 *   y[m,n]  = fl32( float(acc[m,n]) * fl32(gamma_{n/G} / s_m) ).
 * G must divide N (the pages' reshape needs it); G = N is the per-tensor
 * scale. */
void bl_oracle_gamma_groups(const float *W, int64_t N, int64_t K, int64_t G,
                            float *gamma) {
  for (int64_t g = 0; g < N / G; ++g) {
    double S = 0.0;
    for (int64_t n = g * G; n < (g + 1) * G; ++n) {
      double row = 0.0;
      for (int64_t k = 0; k < K; ++k) row += fabs((double)W[n * K + k]);
      S += row;
    }
    float mean = (float)(S / ((double)G * (double)K));
    gamma[g] = mean + 1e-5f;
  }
}

void bl_oracle_ternarize_groups(const float *W, int64_t N, int64_t K, int64_t G,
                                const float *gamma, int8_t *q) {
  for (int64_t n = 0; n < N; ++n) {
    float g = gamma[n / G];
    for (int64_t k = 0; k < K; ++k) {
      float r = W[n * K + k] / g;
      float t = rintf(r);
      if (t > 1.0f) t = 1.0f;
      if (t < -1.0f) t = -1.0f;
      q[n * K + k] = (int8_t)t;
    }
  }
}

void bl_oracle_rescale_groups(const int32_t *acc, const float *gamma, int64_t G,
                              const float *s, int64_t M, int64_t N, float *y) {
  for (int64_t m = 0; m < M; ++m) {
    for (int64_t n = 0; n < N; ++n) {
      float c = gamma[n / G] / s[m];
      float a = (float)acc[m * N + n];
      y[m * N + n] = a * c;
    }
  }
}

/* Fused subln RMSNorm + activation quantisation.
 * [CSDN-2B4T 2, item 3] and [CSDN-0.4GB 1] 归一化方法: subln normalisation
 * sits before the quantised projection; no bias anywhere.
 *   r_t  = fl32( 1 / fl32( sqrt( fl32( fl32(sum_k x_tk^2 / K) + eps ) ) ) )
 *          (sum of squares in fp64, sequential over k)
 *   u_tk = fl32( x_tk * g_k )           (g = 1 when absent)
 *   xq, s_u = quant_act(u)               (per-token absmax, as above)
 *   s_t  = fl32( s_u / r_t )             (the scale of v = u * r_t)
 * Absmax quantisation is invariant under the positive per-token factor r_t,
 * so xq is the code of v = RMSNorm(x) * g and s_t its scale.  r is also
 * returned for the tests.                                                   */
void bl_oracle_rmsnorm_quant_act(const float *x, const float *g, float eps,
                                 int64_t M, int64_t K, int8_t *xq, float *s,
                                 float *r_out, float *u_scratch) {
  for (int64_t m = 0; m < M; ++m) {
    const float *xr = x + m * K;
    double ss = 0.0;
    for (int64_t k = 0; k < K; ++k) ss += (double)xr[k] * (double)xr[k];
    float ms = (float)(ss / (double)K);
    float d = sqrtf(ms + eps);
    float r = 1.0f / d;
    for (int64_t k = 0; k < K; ++k) u_scratch[k] = g ? xr[k] * g[k] : xr[k];
    float su;
    bl_oracle_quant_act(u_scratch, 1, K, xq + m * K, &su);
    s[m] = su / r;
    if (r_out) r_out[m] = r;
  }
}
