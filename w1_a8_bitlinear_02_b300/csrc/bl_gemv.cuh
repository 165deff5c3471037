// Decode GEMV for M <= 4 tokens: y[m, n] = sum_k Wq[n, k] * xq[m, k], rescaled.
//
// The pages place the GPU cost of BitLinear in memory traffic: ternary
// weights are packed several per byte in HBM, loaded on chip and unpacked
// there ("微软AI大模型炸场：0.4GB，CPU就能跑", blog.csdn.net/2401_84494441,
// section 3 "软硬协同", GPU bullet).  This kernel is that idea on sm_103a:
//
//  * A producer warp streams contiguous blocks of packed rows into a ring of
//    shared-memory stages with 1-D bulk copies (cp.async.bulk, mbarrier
//    completion), so each SM keeps ~96 KB of HBM reads in flight without
//    tying up registers.
//  * Each consumer thread owns a fixed set of packed 32-bit words (16
//    weights each) of every row, so its slice of the quantised activations
//    stays in registers for the whole kernel; rows stream past it.
//  * Unpacking costs one AND per 4 weights: for mask i, the bytes of
//    (word & (0x03030303 << 2i)) are the codes c = q + 1 of four weights
//    times 4^i, fed straight to dp4a (unsigned codes x signed activations)
//    into accumulator i; the 4^i factor is removed exactly at the end
//    (each accumulator is a multiple of 4^i).  sum c*x - sum x = sum q*x.
//  * Per-row partial sums are reduced across the threads that share a row
//    with warp shuffles (and shared memory when a row spans warps).
//
// With launch overlap on, the producer starts streaming weights before the
// previous kernel on the stream has finished; everything else waits.
#pragma once

#include <cuda_bf16.h>
#include <cstdint>

#include "bl_pack_quant.cuh"
#include "bl_ptx.cuh"

namespace bl {
namespace gemv {

constexpr int kConsumerWarps = 8;
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kThreads = kConsumers + 32;  // + one producer warp
constexpr int kStages = 3;
constexpr int kStageBytes = 32 * 1024;
constexpr int kSmemBytes = kStages * kStageBytes + 1024;

enum XMode { kXF32 = 0, kXBF16 = 1, kXInt8 = 2 };

struct Params {
  const uint8_t *packed;
  const float *gamma;
  const void *x;        // kXF32 / kXBF16: [M, K] activations
  const int8_t *xq;     // kXInt8: [M, K] codes
  const float *scale;   // kXInt8: [M] scales
  float *y;             // [M, N] (float output)
  int32_t *acc;         // [M, N] (int32 output)
  int64_t N;
  int K;
  int words;            // packed 32-bit words per row (= row_bytes / 4)
  int row_bytes;
  int M;
  int rows_per_cta;
  int stage_rows;       // rows per shared-memory stage (multiple of rows/iter)
  int tpr_log2;         // threads per row = 1 << tpr_log2
};

struct Smem {
  uint64_t full[kStages];
  uint64_t empty[kStages];
  int32_t part[kConsumerWarps][4];
  float fred[kConsumerWarps][4];
  int abort_flag;
};

template <int XM>
__device__ __forceinline__ float load_x(const void *x, int64_t idx) {
  if constexpr (XM == kXF32)
    return static_cast<const float *>(x)[idx];
  else
    return __bfloat162float(static_cast<const __nv_bfloat16 *>(x)[idx]);
}

// MT: tokens held (M <= MT); WPT: packed words per thread per row.
template <int MT, int WPT, int XM, bool OUT_I32>
__global__ void __launch_bounds__(kThreads, 1) gemv_kernel(const Params p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *stages = smem_raw;
  Smem &sm = *reinterpret_cast<Smem *>(smem_raw + kStages * kStageBytes);

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int64_t row0 = static_cast<int64_t>(blockIdx.x) * p.rows_per_cta;
  int64_t nrows = p.N - row0;
  if (nrows > p.rows_per_cta) nrows = p.rows_per_cta;
  if (nrows <= 0) return;  // whole block exits together
  const int n_stages = static_cast<int>((nrows + p.stage_rows - 1) / p.stage_rows);

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&sm.full[s]), 1);
      mbar_init(smem_u32(&sm.empty[s]), kConsumerWarps);
    }
    sm.abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  pdl_launch_dependents();

  if (warp == kConsumerWarps) {
    // ------------------------------------------------ producer warp
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      int issued = 0;
      for (int it = 0; it < n_stages; ++it) {
        const int s = it % kStages;
        if (it >= kStages) {
          if (!mbar_wait(smem_u32(&sm.empty[s]), ((it / kStages) - 1) & 1)) {
            sm.abort_flag = 1;
            break;
          }
          if (*reinterpret_cast<volatile int *>(&sm.abort_flag)) break;
        }
        int64_t rows = nrows - static_cast<int64_t>(it) * p.stage_rows;
        if (rows > p.stage_rows) rows = p.stage_rows;
        const uint32_t bytes = static_cast<uint32_t>(rows) * static_cast<uint32_t>(p.row_bytes);
        const uint32_t fb = smem_u32(&sm.full[s]);
        mbar_arrive_expect_tx(fb, bytes);
        bulk_g2s(smem_u32(stages + s * kStageBytes),
                 p.packed + (row0 + static_cast<int64_t>(it) * p.stage_rows) * p.row_bytes, bytes, fb,
                 pol);
        issued = it + 1;
      }
      // Do not leave while copies into this block's shared memory are in flight.
      for (int it = issued - kStages < 0 ? 0 : issued - kStages; it < issued; ++it)
        mbar_wait(smem_u32(&sm.full[it % kStages]), (it / kStages) & 1);
    }
    return;
  }

  // -------------------------------------------------- consumer warps
  pdl_wait_primary();
  const float gamma = *p.gamma;
  const int tpr = 1 << p.tpr_log2;
  const int lr = tid & (tpr - 1);       // word slot inside the row
  const int rslot = tid >> p.tpr_log2;  // row slot inside an iteration
  const int rpi = kConsumers >> p.tpr_log2;

  // ---- activations of this thread's words, quantised, in registers
  uint32_t xw[MT][WPT][4];
  int xsum[MT];
  float sc[MT];
#pragma unroll
  for (int m = 0; m < MT; ++m) {
    xsum[m] = 0;
    sc[m] = 1.0f;
  }

  if constexpr (XM == kXInt8) {
#pragma unroll
    for (int m = 0; m < MT; ++m) {
      if (m < p.M) sc[m] = p.scale[m];
#pragma unroll
      for (int w = 0; w < WPT; ++w) {
        const int kw = lr + w * tpr;
        uint32_t v[4] = {0u, 0u, 0u, 0u};
        if (m < p.M && kw < p.words) {
          const int64_t base = static_cast<int64_t>(m) * p.K + 16 * kw;
          const int8_t *src = p.xq + base;
          if (16 * kw + 16 <= p.K && ((reinterpret_cast<uintptr_t>(src) & 15u) == 0u)) {
            const uint4 u = *reinterpret_cast<const uint4 *>(src);
            v[0] = u.x; v[1] = u.y; v[2] = u.z; v[3] = u.w;
          } else {
#pragma unroll
            for (int b = 0; b < 16; ++b)
              if (16 * kw + b < p.K)
                v[b >> 2] |= (static_cast<uint32_t>(static_cast<uint8_t>(src[b]))) << (8 * (b & 3));
          }
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          xw[m][w][i] = v[i];
          xsum[m] = dp4a_us(0x01010101u, v[i], xsum[m]);
        }
      }
    }
  } else {
    // per-token absmax over the whole row, reduced over the consumer warps
    float amax[MT];
#pragma unroll
    for (int m = 0; m < MT; ++m) {
      amax[m] = 0.0f;
      if (m < p.M)
        for (int k = tid; k < p.K; k += kConsumers)
          amax[m] = fmaxf(amax[m], fabsf(load_x<XM>(p.x, static_cast<int64_t>(m) * p.K + k)));
      amax[m] = warp_max(amax[m]);
      if (lane == 0) sm.fred[warp][m] = amax[m];
    }
    named_bar(1, kConsumers);
#pragma unroll
    for (int m = 0; m < MT; ++m) {
      float a = sm.fred[0][m];
#pragma unroll
      for (int i = 1; i < kConsumerWarps; ++i) a = fmaxf(a, sm.fred[i][m]);
      sc[m] = act_scale(a);
    }
#pragma unroll
    for (int m = 0; m < MT; ++m) {
#pragma unroll
      for (int w = 0; w < WPT; ++w) {
        const int kw = lr + w * tpr;
        uint32_t v[4] = {0u, 0u, 0u, 0u};
        if (m < p.M && kw < p.words) {
#pragma unroll
          for (int b = 0; b < 16; ++b) {
            const int k = 16 * kw + b;
            if (k < p.K) {
              const int q = quant_one(load_x<XM>(p.x, static_cast<int64_t>(m) * p.K + k), sc[m]);
              v[b >> 2] |= (static_cast<uint32_t>(q) & 0xFFu) << (8 * (b & 3));
            }
          }
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          xw[m][w][i] = v[i];
          xsum[m] = dp4a_us(0x01010101u, v[i], xsum[m]);
        }
      }
    }
  }

  // ---- stream the rows
  const uint32_t stage0 = smem_u32(stages);
  for (int it = 0; it < n_stages; ++it) {
    const int s = it % kStages;
    bool failed = !mbar_wait(smem_u32(&sm.full[s]), (it / kStages) & 1);
    // Warps that share rows meet at named barriers below: decide together.
    if (tpr > 32) failed = named_bar_or(2, kConsumers, failed);
    if (failed) {
      sm.abort_flag = 1;
      break;
    }
    int64_t rows_here = nrows - static_cast<int64_t>(it) * p.stage_rows;
    if (rows_here > p.stage_rows) rows_here = p.stage_rows;
    const uint32_t sbase = stage0 + s * kStageBytes;
    for (int rr = 0; rr < rows_here; rr += rpi) {
      const int r = rr + rslot;
      const bool valid = r < rows_here;
      int tot[MT];
#pragma unroll
      for (int m = 0; m < MT; ++m) tot[m] = 0;
      if (valid) {
        int a0[MT], a1[MT], a2[MT], a3[MT];
#pragma unroll
        for (int m = 0; m < MT; ++m) a0[m] = a1[m] = a2[m] = a3[m] = 0;
        const uint32_t rbase = sbase + static_cast<uint32_t>(r) * p.row_bytes;
#pragma unroll
        for (int w = 0; w < WPT; ++w) {
          const int kw = lr + w * tpr;
          if (kw < p.words) {
            const uint32_t word = lds_u32(rbase + 4u * kw);
            const uint32_t c0 = word & 0x03030303u, c1 = word & 0x0C0C0C0Cu;
            const uint32_t c2 = word & 0x30303030u, c3 = word & 0xC0C0C0C0u;
#pragma unroll
            for (int m = 0; m < MT; ++m) {
              a0[m] = dp4a_us(c0, xw[m][w][0], a0[m]);
              a1[m] = dp4a_us(c1, xw[m][w][1], a1[m]);
              a2[m] = dp4a_us(c2, xw[m][w][2], a2[m]);
              a3[m] = dp4a_us(c3, xw[m][w][3], a3[m]);
            }
          }
        }
#pragma unroll
        for (int m = 0; m < MT; ++m)
          tot[m] = a0[m] + (a1[m] >> 2) + (a2[m] >> 4) + (a3[m] >> 6) - xsum[m];
      }
      // reduce over the tpr threads of the row
      const int width = tpr < 32 ? tpr : 32;
#pragma unroll
      for (int m = 0; m < MT; ++m)
        for (int o = width >> 1; o > 0; o >>= 1) tot[m] += __shfl_xor_sync(0xffffffffu, tot[m], o);
      if (tpr > 32) {
        if (lane == 0) {
#pragma unroll
          for (int m = 0; m < MT; ++m) sm.part[warp][m] = tot[m];
        }
        named_bar(1, kConsumers);
        if (lr == 0) {
          const int w0 = warp, nw = tpr >> 5;
#pragma unroll
          for (int m = 0; m < MT; ++m) {
            int v = 0;
            for (int i = 0; i < nw; ++i) v += sm.part[w0 + i][m];
            tot[m] = v;
          }
        }
        named_bar(1, kConsumers);
      }
      if (valid && lr == 0) {
        const int64_t n = row0 + static_cast<int64_t>(it) * p.stage_rows + r;
#pragma unroll
        for (int m = 0; m < MT; ++m) {
          if (m < p.M) {
            if constexpr (OUT_I32)
              p.acc[static_cast<int64_t>(m) * p.N + n] = tot[m];
            else
              p.y[static_cast<int64_t>(m) * p.N + n] =
                  __fdiv_rn(__fmul_rn(static_cast<float>(tot[m]), gamma), sc[m]);
          }
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&sm.empty[s]));
  }
}

}  // namespace gemv
}  // namespace bl
