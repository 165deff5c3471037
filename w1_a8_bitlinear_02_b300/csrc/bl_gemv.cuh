// Decode GEMV for M <= 8 tokens: y[m, n] = sum_k Wq[n, k] * xq[m, k], rescaled.
//
// The pages place the GPU cost of BitLinear in memory traffic: ternary
// weights are packed several per byte in HBM, loaded on chip and unpacked
// there ("微软AI大模型炸场：0.4GB，CPU就能跑", blog.csdn.net/2401_84494441,
// section 3 "软硬协同", GPU bullet).  On sm_103a:
//
//  * One elected thread streams each block's contiguous run of packed rows
//    into a ring of shared-memory stages with 1-D bulk copies (cp.async.bulk,
//    mbarrier completion): up to ~190 KB in flight per SM without any
//    per-thread copy instructions or registers.  With launch overlap on, it
//    starts before the previous kernel on the stream has finished.
//  * A warp owns whole rows.  Lane l holds the activation codes of the 8-byte
//    units (32 weights) l, l + 32, ... of its chunk of K in registers, so a
//    row costs each lane a few 8-byte shared loads and the row's sum is one
//    warp reduction.  Very long rows are split over G warps whose partial
//    sums meet in shared memory (a per-row counter picks the last arriver,
//    which writes the output; no block barriers).
//  * Unpacking: for M <= 2, one AND per 4 weights -- the bytes of
//    (word & (0x03030303 << 2i)) are the codes c = q + 1 of four weights times
//    4^i, fed to dp4a (unsigned codes x signed activations) into accumulator
//    i; the 4^i factor is removed exactly at the end (each accumulator is a
//    multiple of 4^i).  For more tokens the codes are shifted down once per
//    word and shared by all tokens.  sum c*x - X = sum q*x, with
//    X = sum_k xq[m, k] from the quantisation pass.
//  * The activation rows are quantised once per block into shared memory
//    (per-token absmax, block reduction), then each warp pulls its chunk.
#pragma once

#include <cuda_bf16.h>
#include <cstdint>

#include "bl_pack_quant.cuh"
#include "bl_ptx.cuh"

namespace bl {
namespace gemv {

constexpr int kMaxStages = 6;
constexpr int kStageBytes = 64 * 1024;  // upper bound of one stage
constexpr int kMaxSplitRows = 32;       // rows per stage when rows are split over warps
constexpr int kSmemFixed = 8 * 1024;    // barriers, reductions, split-row partials

enum XMode { kXF32 = 0, kXBF16 = 1, kXInt8 = 2 };

struct Params {
  const uint8_t *packed;
  const float *gamma;
  const void *x;        // kXF32 / kXBF16: [M, K] activations
  const int8_t *xq;     // kXInt8: [M, K] codes
  const float *scale;   // kXInt8: [M] scales
  OutSpec out;          // y [M, N] (float output)
  int32_t *acc;         // [M, N] (int32 output)
  int64_t N;
  int K;
  int kp;               // K padded to 64: activation code row length in smem
  int units;            // 8-byte units per packed row (= row_bytes / 8)
  int row_bytes;
  int M;
  int rows_per_cta;
  int stage_rows;       // rows per stage (<= kMaxSplitRows when split > 1)
  int stage_bytes;      // stage_rows * row_bytes rounded up to 128
  int nstages;          // ring depth (<= kMaxStages)
  int split_log2;       // G = warps per row
  int chunk;            // units per warp's chunk of a row (ceil(units / G))
  int wait_prior;       // 1: inputs may come from the previous kernel (wait for it)
  int act;              // activation before quantisation (kActNone / kActRelu2)
};

struct Smem {
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];
  float fred[16][8];
  int32_t xsum[16][8];
  int32_t part[kMaxStages][kMaxSplitRows][8];
  uint32_t cnt[kMaxStages][kMaxSplitRows];
  int abort_flag;
};
static_assert(sizeof(Smem) <= kSmemFixed, "fixed shared-memory region");

template <int XM>
__device__ __forceinline__ float load_x(const void *x, int64_t idx) {
  if constexpr (XM == kXF32)
    return static_cast<const float *>(x)[idx];
  else
    return __bfloat162float(static_cast<const __nv_bfloat16 *>(x)[idx]);
}

template <int XM>
__device__ __forceinline__ void load8x(const void *x, int64_t idx, float (&v)[8]) {
  if constexpr (XM == kXF32)
    load8(static_cast<const float *>(x) + idx, v);
  else
    load8(static_cast<const __nv_bfloat16 *>(x) + idx, v);
}

__device__ __forceinline__ uint2 lds_u64(uint32_t addr) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
  return v;
}

// One row's sum over this lane's units (lbase: the lane's first unit; unit u
// at + 256 u).  FULL: every unit exists; otherwise unit u is read at + uoff[u],
// which points back at an existing unit of the row where unit u does not
// exist: its activation codes are zero, so it adds nothing, and the loop has
// no per-unit branch (a branch per unit serialises the loads and measured
// more than twice as slow per row on B300).
//   MT <= 2: the bytes of (word & (3 << 2i)) are codes x 4^i; dp4a into
//   accumulator i and divide by 4^i exactly at the end.
//   MT > 2: the codes are shifted down once per word and shared by the tokens.
template <int MT, int UPT, bool FULL>
__device__ __forceinline__ void row_dot(uint32_t lbase, const uint32_t (&uoff)[UPT], const uint32_t (&xa)[MT][UPT][8],
                                        int (&tot)[MT]) {
  if constexpr (MT <= 2) {
    int a0[MT], a1[MT], a2[MT], a3[MT];
#pragma unroll
    for (int m = 0; m < MT; ++m) a0[m] = a1[m] = a2[m] = a3[m] = 0;
#pragma unroll
    for (int u = 0; u < UPT; ++u) {
      const uint2 wv = lds_u64(lbase + (FULL ? 256u * u : uoff[u]));
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const uint32_t word = h ? wv.y : wv.x;
        const uint32_t c0 = word & 0x03030303u, c1 = word & 0x0C0C0C0Cu;
        const uint32_t c2 = word & 0x30303030u, c3 = word & 0xC0C0C0C0u;
#pragma unroll
        for (int m = 0; m < MT; ++m) {
          a0[m] = dp4a_us(c0, xa[m][u][4 * h + 0], a0[m]);
          a1[m] = dp4a_us(c1, xa[m][u][4 * h + 1], a1[m]);
          a2[m] = dp4a_us(c2, xa[m][u][4 * h + 2], a2[m]);
          a3[m] = dp4a_us(c3, xa[m][u][4 * h + 3], a3[m]);
        }
      }
    }
#pragma unroll
    for (int m = 0; m < MT; ++m) tot[m] = a0[m] + (a1[m] >> 2) + (a2[m] >> 4) + (a3[m] >> 6);
  } else {
    int a[MT];
#pragma unroll
    for (int m = 0; m < MT; ++m) a[m] = 0;
#pragma unroll
    for (int u = 0; u < UPT; ++u) {
      const uint2 wv = lds_u64(lbase + (FULL ? 256u * u : uoff[u]));
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const uint32_t word = h ? wv.y : wv.x;
        const uint32_t c0 = word & 0x03030303u, c1 = (word >> 2) & 0x03030303u;
        const uint32_t c2 = (word >> 4) & 0x03030303u, c3 = (word >> 6) & 0x03030303u;
#pragma unroll
        for (int m = 0; m < MT; ++m) {
          a[m] = dp4a_us(c0, xa[m][u][4 * h + 0], a[m]);
          a[m] = dp4a_us(c1, xa[m][u][4 * h + 1], a[m]);
          a[m] = dp4a_us(c2, xa[m][u][4 * h + 2], a[m]);
          a[m] = dp4a_us(c3, xa[m][u][4 * h + 3], a[m]);
        }
      }
    }
#pragma unroll
    for (int m = 0; m < MT; ++m) tot[m] = a[m];
  }
}

// MT: tokens held (M <= MT); UPT: 8-byte units per lane; CW: consumer warps.
template <int MT, int UPT, int XM, bool OUT_I32, int CW>
__global__ void __launch_bounds__((CW + 1) * 32, 1) gemv_kernel(const Params p) {
  constexpr int kConsumers = CW * 32;
  extern __shared__ __align__(128) uint8_t smem_raw[];
  Smem &sm = *reinterpret_cast<Smem *>(smem_raw);
  const uint32_t ring = smem_u32(smem_raw + kSmemFixed);
  const uint32_t xs = ring + static_cast<uint32_t>(p.nstages * p.stage_bytes);  // [M][kp] codes

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t row0 = static_cast<int64_t>(blockIdx.x) * p.rows_per_cta;
  int64_t nrows64 = p.N - row0;
  if (nrows64 > p.rows_per_cta) nrows64 = p.rows_per_cta;
  const int nrows = static_cast<int>(nrows64);
  const int n_iters = (nrows + p.stage_rows - 1) / p.stage_rows;
  const int S = p.nstages;

  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(smem_u32(&sm.full[s]), 1);
      mbar_init(smem_u32(&sm.empty[s]), CW);
    }
    sm.abort_flag = 0;
    fence_barrier_init();
  }
  for (int i = tid; i < kMaxStages * kMaxSplitRows; i += blockDim.x) {
    (&sm.cnt[0][0])[i] = 0u;
#pragma unroll
    for (int m = 0; m < 8; ++m) (&sm.part[0][0][0])[i * 8 + m] = 0;
  }
  __syncthreads();

  if (warp == CW) {
    // ------------------------------------------------ producer warp
    pdl_launch_dependents();
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      int issued = 0;
      for (int it = 0; it < n_iters; ++it) {
        const int s = it % S;
        if (it >= S) {
          if (!mbar_wait(smem_u32(&sm.empty[s]), ((it / S) - 1) & 1)) {
            sm.abort_flag = 1;
            break;
          }
          if (*reinterpret_cast<volatile int *>(&sm.abort_flag)) break;
        }
        int rows = nrows - it * p.stage_rows;
        if (rows > p.stage_rows) rows = p.stage_rows;
        const uint32_t bytes = static_cast<uint32_t>(rows) * static_cast<uint32_t>(p.row_bytes);
        const uint32_t fb = smem_u32(&sm.full[s]);
        mbar_arrive_expect_tx(fb, bytes);
        bulk_g2s(ring + s * p.stage_bytes,
                 p.packed + (row0 + static_cast<int64_t>(it) * p.stage_rows) * p.row_bytes, bytes, fb, pol);
        issued = it + 1;
      }
      // Do not leave while copies into this block's shared memory are in flight.
      for (int it = issued - S < 0 ? 0 : issued - S; it < issued; ++it)
        mbar_wait(smem_u32(&sm.full[it % S]), (it / S) & 1);
    }
    return;
  }

  // -------------------------------------------------- consumer warps
  // gamma is a static input like the packed weights: read it before waiting.
  const float gamma = OUT_I32 ? 1.0f : __ldg(p.gamma);
  pdl_launch_dependents();
  if (p.wait_prior) pdl_wait_primary();

  // ---- activation codes of the M tokens into shared memory, with
  // X_m = sum_k xq[m, k] (turns sum c*x into sum q*x at the end)
  float sc[MT];
#pragma unroll
  for (int m = 0; m < MT; ++m) sc[m] = 1.0f;
  if constexpr (XM == kXInt8) {
    const bool vec = (reinterpret_cast<uintptr_t>(p.xq) & 15u) == 0u && (p.K % 16) == 0;
#pragma unroll
    for (int m = 0; m < MT; ++m) {
      int part = 0;
      if (m < p.M) {
        const int8_t *src = p.xq + static_cast<int64_t>(m) * p.K;
        const uint32_t xrow = xs + static_cast<uint32_t>(m * p.kp);
        const int nv = vec ? p.K / 16 : 0;
        for (int c = tid; c < nv; c += kConsumers) {
          const uint4 v = __ldg(reinterpret_cast<const uint4 *>(src) + c);
          sts_u128(xrow + 16 * c, v.x, v.y, v.z, v.w);
          part = dp4a_us(0x01010101u, v.x, part);
          part = dp4a_us(0x01010101u, v.y, part);
          part = dp4a_us(0x01010101u, v.z, part);
          part = dp4a_us(0x01010101u, v.w, part);
        }
        for (int k = 16 * nv + tid; k < p.kp; k += kConsumers) {
          const int q = k < p.K ? static_cast<int>(src[k]) : 0;
          sts_u8(xrow + k, static_cast<uint32_t>(q) & 0xFFu);
          part += q;
        }
        if constexpr (!OUT_I32) sc[m] = __ldg(p.scale + m);
      }
      part = __reduce_add_sync(0xffffffffu, part);
      if (lane == 0) sm.xsum[warp][m] = part;
    }
  } else {
    // per-token absmax over 8-element vectors strided over K, block reduction,
    // then the codes.  When a thread's vectors of all tokens fit in JM
    // registers each they are all requested at once and kept for the second
    // step: one round trip to memory; else a second pass over the same
    // vectors (L1 hits).
    const bool vec = (reinterpret_cast<uintptr_t>(p.x) & 15u) == 0u && (p.K % 8) == 0;
    const int nv = vec ? p.K / 8 : 0;
    // A row of units <= 32 UPT (one warp per row) has K / 8 <= 4 UPT vectors,
    // at most (UPT + 1) / 2 per thread of 8 consumer warps.
    constexpr int JM = (UPT + 1) / 2 / MT > 0 ? (UPT + 1) / 2 / MT : 1;  // vectors per token in registers
    const bool in_regs = nv <= JM * kConsumers;
    float xv[MT][JM][8];
    if (in_regs) {
#pragma unroll
      for (int m = 0; m < MT; ++m)
#pragma unroll
        for (int j = 0; j < JM; ++j) {
          const int c = tid + j * kConsumers;
          if (m < p.M && c < nv) {
            load8x<XM>(p.x, static_cast<int64_t>(m) * p.K + 8 * c, xv[m][j]);
          } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) xv[m][j][e] = 0.0f;
          }
        }
      // the activation after every load is in flight (relu2(0) = 0)
      if (p.act == kActRelu2)
#pragma unroll
        for (int m = 0; m < MT; ++m)
#pragma unroll
          for (int j = 0; j < JM; ++j)
#pragma unroll
            for (int e = 0; e < 8; ++e) xv[m][j][e] = relu2f(xv[m][j][e]);
    }
#pragma unroll
    for (int m = 0; m < MT; ++m) {
      float a = 0.0f;
      if (m < p.M) {
        const int64_t row = static_cast<int64_t>(m) * p.K;
        if (in_regs) {
#pragma unroll
          for (int j = 0; j < JM; ++j)
#pragma unroll
            for (int e = 0; e < 8; ++e) a = fmaxf(a, fabsf(xv[m][j][e]));
        } else {
          if (p.act == kActRelu2) {
#pragma unroll 2
            for (int c = tid; c < nv; c += kConsumers) {
              float v[8];
              load8x<XM>(p.x, row + 8 * c, v);
#pragma unroll
              for (int j = 0; j < 8; ++j) a = fmaxf(a, relu2f(v[j]));
            }
          } else {
#pragma unroll 2
            for (int c = tid; c < nv; c += kConsumers) {
              float v[8];
              load8x<XM>(p.x, row + 8 * c, v);
#pragma unroll
              for (int j = 0; j < 8; ++j) a = fmaxf(a, fabsf(v[j]));
            }
          }
        }
        for (int k = 8 * nv + tid; k < p.K; k += kConsumers) {
          const float v = load_x<XM>(p.x, row + k);
          a = fmaxf(a, fabsf(p.act == kActRelu2 ? relu2f(v) : v));
        }
      }
      a = warp_max_nonneg(a);
      if (lane == 0) sm.fred[warp][m] = a;
    }
    named_bar(1, kConsumers);
#pragma unroll
    for (int m = 0; m < MT; ++m) {
      float a = sm.fred[0][m];
#pragma unroll
      for (int i = 1; i < CW; ++i) a = fmaxf(a, sm.fred[i][m]);
      sc[m] = act_scale(a);
    }
#pragma unroll
    for (int m = 0; m < MT; ++m) {
      int part = 0;
      if (m < p.M) {
        const int64_t row = static_cast<int64_t>(m) * p.K;
        const uint32_t xrow = xs + static_cast<uint32_t>(m * p.kp);
        auto put8 = [&](int c, const float (&v)[8]) {
          uint32_t lo = 0, hi = 0;
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int q0 = quant_one(v[j], sc[m]), q1 = quant_one(v[j + 4], sc[m]);
            part += q0 + q1;
            lo |= (static_cast<uint32_t>(q0) & 0xFFu) << (8 * j);
            hi |= (static_cast<uint32_t>(q1) & 0xFFu) << (8 * j);
          }
          sts_u64(xrow + 8 * c, lo, hi);
        };
        if (in_regs) {
#pragma unroll
          for (int j = 0; j < JM; ++j) {
            const int c = tid + j * kConsumers;
            if (c < nv) put8(c, xv[m][j]);
          }
        } else {
#pragma unroll 2
          for (int c = tid; c < nv; c += kConsumers) {
            float v[8];
            load8x<XM>(p.x, row + 8 * c, v);
            if (p.act == kActRelu2)
#pragma unroll
              for (int e = 0; e < 8; ++e) v[e] = relu2f(v[e]);
            put8(c, v);
          }
        }
        for (int k = 8 * nv + tid; k < p.kp; k += kConsumers) {
          float v = k < p.K ? load_x<XM>(p.x, row + k) : 0.0f;
          if (p.act == kActRelu2) v = relu2f(v);
          const int q = k < p.K ? quant_one(v, sc[m]) : 0;
          part += q;
          sts_u8(xrow + k, static_cast<uint32_t>(q) & 0xFFu);
        }
      }
      part = __reduce_add_sync(0xffffffffu, part);
      if (lane == 0) sm.xsum[warp][m] = part;
    }
  }
  named_bar(1, kConsumers);

  // the token's output scale c_m = gamma / s_m (one true division per token)
  float cm[MT];
  int xtot[MT];
#pragma unroll
  for (int m = 0; m < MT; ++m) {
    cm[m] = __fdiv_rn(gamma, sc[m]);
    int v = 0;
#pragma unroll
    for (int i = 0; i < CW; ++i) v += sm.xsum[i][m];
    xtot[m] = v;
  }

  // ---- this lane's activation codes: 32 per 8-byte weight unit of its chunk
  const int G = 1 << p.split_log2;
  const int chunk_id = warp & (G - 1);
  const int row_slot = warp >> p.split_log2;
  // A row split over more warps than the block has cannot be covered: report
  // it and do no row work (the launch plan guarantees G <= CW).
  const bool split_ok = G <= CW;
  if (!split_ok && tid == 0) atomicOr(&g_dev_error, kDevErrConfig);
  const int row_step = split_ok ? (CW >> p.split_log2) : 1;
  const int ubase = chunk_id * p.chunk;
  int uend = ubase + p.chunk;
  if (uend > p.units) uend = p.units;
  uint32_t xa[MT][UPT][8];
#pragma unroll
  for (int m = 0; m < MT; ++m) {
#pragma unroll
    for (int u = 0; u < UPT; ++u) {
      const int unit = ubase + lane + 32 * u;
      uint4 a = make_uint4(0u, 0u, 0u, 0u), b = a;
      if (m < p.M && unit < uend) {
        const uint32_t at = xs + static_cast<uint32_t>(m * p.kp + 32 * unit);
        a = lds_u128(at);
        b = lds_u128(at + 16);
      }
      xa[m][u][0] = a.x; xa[m][u][1] = a.y; xa[m][u][2] = a.z; xa[m][u][3] = a.w;
      xa[m][u][4] = b.x; xa[m][u][5] = b.y; xa[m][u][6] = b.z; xa[m][u][7] = b.w;
    }
  }

  // This lane's units are ubase + lane + 32 u.  When every lane's UPT units
  // lie inside the chunk the row loop uses fixed offsets; otherwise a unit
  // past the chunk is read at the chunk's first unit (codes zero, see row_dot),
  // and so is every unit of a lane that starts past it.
  const bool lane_in = ubase + lane < uend;
  const uint32_t lane_addr = 8u * static_cast<uint32_t>(lane_in ? ubase + lane : ubase);
  const bool all_in = ubase + 32 * UPT <= uend;
  uint32_t uoff[UPT];
#pragma unroll
  for (int u = 0; u < UPT; ++u) uoff[u] = (lane_in && ubase + lane + 32 * u < uend) ? 256u * u : 0u;

  // ---- stream the rows
  for (int it = 0; it < n_iters; ++it) {
    const int s = it % S;
    if (!mbar_wait(smem_u32(&sm.full[s]), (it / S) & 1)) {
      sm.abort_flag = 1;
      break;
    }
    int rows_here = nrows - it * p.stage_rows;
    if (rows_here > p.stage_rows) rows_here = p.stage_rows;
    const uint32_t sbase = ring + s * p.stage_bytes;
    for (int r = split_ok ? row_slot : rows_here; r < rows_here; r += row_step) {
      // this lane's units: lane_base + 256 u; only the last can fall past the chunk
      const uint32_t lbase = sbase + static_cast<uint32_t>(r) * p.row_bytes + lane_addr;
      int tot[MT];
      if (all_in)
        row_dot<MT, UPT, true>(lbase, uoff, xa, tot);
      else
        row_dot<MT, UPT, false>(lbase, uoff, xa, tot);
#pragma unroll
      for (int m = 0; m < MT; ++m) tot[m] = __reduce_add_sync(0xffffffffu, tot[m]);
      if (lane == 0) {
        bool write = true;
        if (G > 1) {  // meet the row's other chunks in shared memory
#pragma unroll
          for (int m = 0; m < MT; ++m)
            if (m < p.M) atomicAdd(&sm.part[s][r][m], tot[m]);
          __threadfence_block();
          write = atomicAdd(&sm.cnt[s][r], 1u) == static_cast<uint32_t>(G - 1);
          if (write) {
            __threadfence_block();
#pragma unroll
            for (int m = 0; m < MT; ++m)
              if (m < p.M) tot[m] = atomicExch(&sm.part[s][r][m], 0);
            sm.cnt[s][r] = 0u;
          }
        }
        if (write) {
          const int64_t n = row0 + static_cast<int64_t>(it) * p.stage_rows + r;
#pragma unroll
          for (int m = 0; m < MT; ++m) {
            if (m < p.M) {
              const int q = tot[m] - xtot[m];  // sum (c - 1) x = sum q x
              if constexpr (OUT_I32)
                p.acc[static_cast<int64_t>(m) * p.N + n] = q;
              else
                put_y(p.out, static_cast<int64_t>(m) * p.N + n,
                      __fmul_rn(static_cast<float>(q), p.out.gvec ? group_scale(p.out, n, sc[m]) : cm[m]));
            }
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
