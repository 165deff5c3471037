// Decode chain: a sequence of M = 1 BitLinear forwards in one persistent
// launch, call i + 1 reading its input only after call i has written its
// output (so an input may be an earlier call's output).
//
// A decode step runs the projections of every layer one after another
// ("BitNet b1.58 2B4T" architecture: QKV, O, FFN up, FFN down per layer;
// "20亿参数仅0.4GB…「原生1.58bit」大模型", blog.csdn.net/soaring_casia,
// section 2).  As separate launches each call pays a kernel boundary (the
// next kernel may read the previous one's output only after the whole grid
// has finished and flushed) although its packed weights -- static inputs --
// are a fraction of a microsecond of HBM time.  Here one block per SM stays
// resident for the whole chain:
//   * its producer thread streams the block's rows of every call, call after
//     call, into one bulk-copy ring: the weights of later calls arrive while
//     earlier calls compute, limited only by the ring's size;
//   * the consumer warps run the calls in order; between dependent calls the
//     blocks meet at a software grid barrier (one release-add per block on a
//     counter, acquire-spin until every block has arrived), then quantise the
//     new input and run their rows as the GEMV does (masked dp4a on the
//     packed codes, exact int32 sums, y = fl32(acc * fl32(gamma / s))).
// All blocks must be resident at once (they wait for each other): the launch
// is cooperative, one block per SM.
#pragma once

#include <cuda_bf16.h>
#include <cstdint>

#include "bl_gemv.cuh"
#include "bl_pack_quant.cuh"
#include "bl_ptx.cuh"

namespace bl {
namespace chain {

constexpr int kMaxCalls = 128;
constexpr int kCW = 8;                    // consumer warps
constexpr int kThreads = (kCW + 1) * 32;  // + one producer warp
constexpr int kUPT = 8;                   // 8-byte units per lane: rows up to 256 units (K <= 8192)
constexpr int kMaxK = 32 * kUPT * 32;     // 8192
constexpr int kStageBytes = 32 * 1024;
constexpr int kStages = 6;
constexpr int kJM = 4;                    // x vectors of 8 per consumer thread (8192 / 8 / 256)
constexpr int kSmemFixed = 8192;  // barriers, reductions and the call table
constexpr int kSmemBytes = kSmemFixed + kStages * kStageBytes + kMaxK;  // + activation codes

struct Call {
  const uint8_t *packed;  // [N, 16 * ceil(K / 64)]
  const float *gamma;
  const void *x;          // [K] f32 or bf16
  float *y;               // [N]
  int N, K;
  int xbf16;              // 1: x is bf16
  int act;                // kActNone / kActRelu2
  int wait_prev;          // 1: x may be written by earlier calls (grid barrier first)
};

struct Params {
  int n;                  // calls
  unsigned *bar;          // grid-barrier counter, zero at launch
  Call c[kMaxCalls];
};

struct Smem {
  uint64_t full[kStages];
  uint64_t empty[kStages];
  float fred[kCW];
  int xsum[kCW];
  int abort_flag;
  Call calls[kMaxCalls];  // the parameters, copied once: indexed reads of the
                          // parameter space go through the constant cache
};
static_assert(sizeof(Call) % 4 == 0, "call table copied in words");
static_assert(sizeof(Smem) <= kSmemFixed, "fixed shared-memory region");

__device__ __forceinline__ void red_release_add(unsigned *p, unsigned v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ unsigned ld_acquire(const unsigned *p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// One row's code-weighted sum over this lane's first U units (unit u at
// lbase + 256 u), as the GEMV's masked dp4a loop; FULL: all U units exist,
// otherwise unit u is read at lbase + uoff[u], an existing unit of the row
// where unit u does not exist (its activation codes are zero: it adds
// nothing, and the loop needs no per-unit branch).  U is the call's
// ceil(units / 32), so short rows do not pay for the longest row's loop.
template <int U, bool FULL>
__device__ __forceinline__ int row_sum(uint32_t lbase, const uint32_t (&uoff)[kUPT], const uint32_t (&xa)[kUPT][8]) {
  int a0 = 0, a1 = 0, a2 = 0, a3 = 0;
#pragma unroll
  for (int u = 0; u < U; ++u) {
    const uint2 wv = gemv::lds_u64(lbase + (FULL ? 256u * u : uoff[u]));
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint32_t word = h ? wv.y : wv.x;
      a0 = dp4a_us(word & 0x03030303u, xa[u][4 * h + 0], a0);
      a1 = dp4a_us(word & 0x0C0C0C0Cu, xa[u][4 * h + 1], a1);
      a2 = dp4a_us(word & 0x30303030u, xa[u][4 * h + 2], a2);
      a3 = dp4a_us(word & 0xC0C0C0C0u, xa[u][4 * h + 3], a3);
    }
  }
  return a0 + (a1 >> 2) + (a2 >> 4) + (a3 >> 6);
}

template <int U>
__device__ __forceinline__ void stage_rows(uint32_t sbase, int nr, int rb, uint32_t laddr, int warp,
                                           const uint32_t (&uoff)[kUPT], bool full,
                                           const uint32_t (&xa)[kUPT][8], int xtot, float cm, float *y,
                                           int lane) {
  for (int r = warp; r < nr; r += kCW) {
    const uint32_t lbase = sbase + static_cast<uint32_t>(r * rb) + laddr;
    int t = full ? row_sum<U, true>(lbase, uoff, xa) : row_sum<U, false>(lbase, uoff, xa);
    t = __reduce_add_sync(0xffffffffu, t);
    if (lane == 0) y[r] = __fmul_rn(static_cast<float>(t - xtot), cm);
  }
}

// Rows of call c owned by this block: [r0, r0 + rows).
__device__ __forceinline__ void block_rows(const Call &c, int &r0, int &rows) {
  const int rpc = (c.N + static_cast<int>(gridDim.x) - 1) / static_cast<int>(gridDim.x);
  r0 = static_cast<int>(blockIdx.x) * rpc;
  rows = c.N - r0 < rpc ? c.N - r0 : rpc;
  if (rows < 0) rows = 0;
}
__device__ __forceinline__ int row_bytes_of(int K) { return ((K + 63) / 64) * 16; }

__global__ void __launch_bounds__(kThreads, 1) chain_kernel(const __grid_constant__ Params p) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  Smem &sm = *reinterpret_cast<Smem *>(smem_raw);
  const uint32_t ring = smem_u32(smem_raw + kSmemFixed);
  const uint32_t xs = ring + kStages * kStageBytes;  // activation codes of the current call
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&sm.full[s]), 1);
      mbar_init(smem_u32(&sm.empty[s]), kCW);
    }
    sm.abort_flag = 0;
    fence_barrier_init();
  }
  {
    const uint32_t *src = reinterpret_cast<const uint32_t *>(p.c);
    uint32_t *dst = reinterpret_cast<uint32_t *>(sm.calls);
    const int words = p.n * static_cast<int>(sizeof(Call) / 4);
    for (int w = tid; w < words; w += kThreads) dst[w] = src[w];
  }
  __syncthreads();
  volatile int *abort_flag = &sm.abort_flag;

  if (warp == kCW) {
    // ------------------------------------------------ producer: every call's rows, in order
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      int i = 0, issued = 0;
      bool go = true;
      for (int ci = 0; ci < p.n && go; ++ci) {
        const Call &c = sm.calls[ci];
        int r0, rows;
        block_rows(c, r0, rows);
        const int rb = row_bytes_of(c.K);
        const int sr = kStageBytes / rb;
        for (int q = 0; q < rows; q += sr, ++i) {
          const int s = i % kStages;
          if (i >= kStages && (!mbar_wait(smem_u32(&sm.empty[s]), ((i / kStages) - 1) & 1) || *abort_flag)) {
            *abort_flag = 1;
            go = false;
            break;
          }
          const int nr = rows - q < sr ? rows - q : sr;
          const uint32_t bytes = static_cast<uint32_t>(nr * rb);
          const uint32_t fb = smem_u32(&sm.full[s]);
          mbar_arrive_expect_tx(fb, bytes);
          bulk_g2s(ring + s * kStageBytes, c.packed + static_cast<int64_t>(r0 + q) * rb, bytes, fb, pol);
          issued = i + 1;
        }
      }
      // no copy into this block's shared memory may be in flight at exit
      for (int j = issued - kStages < 0 ? 0 : issued - kStages; j < issued; ++j)
        mbar_wait(smem_u32(&sm.full[j % kStages]), (j / kStages) & 1);
    }
    return;
  }

  // -------------------------------------------------- consumers
  constexpr int kC = kCW * 32;
  int i = 0;  // ring stage counter, in the producer's order
  for (int ci = 0; ci < p.n; ++ci) {
    const Call c = sm.calls[ci];
    const float gam = __ldg(c.gamma);  // static input: fetched while the barrier is awaited
    int r0, rows;
    block_rows(c, r0, rows);
    const int rb = row_bytes_of(c.K);
    const int units = rb / 8;
    const int kp = rb * 4;
    const int sr = kStageBytes / rb;

    // wait until every block has finished the previous call
    if (ci > 0 && c.wait_prev) {
      bool late = false;
      if (tid == 0) {
        const unsigned target = static_cast<unsigned>(ci) * gridDim.x;
        const long long t0 = clock64();
        while (ld_acquire(p.bar) < target) {
          if (clock64() - t0 > kWaitLimitCycles) {
            atomicOr(&g_dev_error, kDevErrTimeout);
            late = true;
            break;
          }
        }
      }
      if (named_bar_or(1, kC, late)) *abort_flag = 1;
    }

    if (rows > 0) {
      // ---- x -> codes in shared memory, X = sum of codes, s, c = gamma / s
      // (x may have been written by other blocks: loads bypass L1)
      const int nv = c.K / 8;
      const bool vec = (c.K % 8) == 0 &&
                       (reinterpret_cast<uintptr_t>(c.x) & 15u) == 0u;
      float xv[kJM][8];
      float a = 0.0f;
      if (vec) {
#pragma unroll
        for (int j = 0; j < kJM; ++j) {
          const int v = tid + j * kC;
          if (v < nv) {
            if (c.xbf16) {
              const uint4 u = __ldcg(reinterpret_cast<const uint4 *>(c.x) + v);
              const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                xv[j][2 * e] = __uint_as_float(w[e] << 16);
                xv[j][2 * e + 1] = __uint_as_float(w[e] & 0xFFFF0000u);
              }
            } else {
              const float4 f0 = __ldcg(reinterpret_cast<const float4 *>(c.x) + 2 * v);
              const float4 f1 = __ldcg(reinterpret_cast<const float4 *>(c.x) + 2 * v + 1);
              xv[j][0] = f0.x; xv[j][1] = f0.y; xv[j][2] = f0.z; xv[j][3] = f0.w;
              xv[j][4] = f1.x; xv[j][5] = f1.y; xv[j][6] = f1.z; xv[j][7] = f1.w;
            }
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              if (c.act == kActRelu2) xv[j][e] = relu2f(xv[j][e]);
              a = fmaxf(a, fabsf(xv[j][e]));
            }
          }
        }
      }
      auto load_one = [&](int k) -> float {
        float v = c.xbf16 ? __bfloat162float(__ldcg(static_cast<const __nv_bfloat16 *>(c.x) + k))
                          : __ldcg(static_cast<const float *>(c.x) + k);
        return c.act == kActRelu2 ? relu2f(v) : v;
      };
      for (int k = (vec ? 8 * nv : 0) + tid; k < c.K; k += kC) a = fmaxf(a, fabsf(load_one(k)));
      a = warp_max_nonneg(a);
      if (lane == 0) sm.fred[warp] = a;
      named_bar(1, kC);
      a = sm.fred[0];
#pragma unroll
      for (int w = 1; w < kCW; ++w) a = fmaxf(a, sm.fred[w]);
      const float s = act_scale(a);
      int part = 0;
      if (vec) {
#pragma unroll
        for (int j = 0; j < kJM; ++j) {
          const int v = tid + j * kC;
          if (v < nv) {
            uint32_t lo = 0, hi = 0;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int q0 = quant_one(xv[j][e], s), q1 = quant_one(xv[j][e + 4], s);
              part += q0 + q1;
              lo |= (static_cast<uint32_t>(q0) & 0xFFu) << (8 * e);
              hi |= (static_cast<uint32_t>(q1) & 0xFFu) << (8 * e);
            }
            sts_u64(xs + 8 * v, lo, hi);
          }
        }
      }
      for (int k = (vec ? 8 * nv : 0) + tid; k < kp; k += kC) {
        const int q = k < c.K ? quant_one(load_one(k), s) : 0;
        part += q;
        sts_u8(xs + k, static_cast<uint32_t>(q) & 0xFFu);
      }
      part = __reduce_add_sync(0xffffffffu, part);
      if (lane == 0) sm.xsum[warp] = part;
      named_bar(1, kC);
      int xtot = 0;
#pragma unroll
      for (int w = 0; w < kCW; ++w) xtot += sm.xsum[w];
      const float cm = __fdiv_rn(gam, s);

      // ---- this lane's activation codes: units lane + 32 u
      uint32_t xa[kUPT][8];
      uint32_t uoff[kUPT];
      const bool lane_in = lane < units;  // otherwise every unit is read at unit 0
      const uint32_t laddr = lane_in ? 8u * lane : 0u;
#pragma unroll
      for (int u = 0; u < kUPT; ++u) {
        const int unit = lane + 32 * u;
        uint4 lo4 = make_uint4(0u, 0u, 0u, 0u), hi4 = lo4;
        uoff[u] = 0u;
        if (unit < units) {
          lo4 = lds_u128(xs + 32 * unit);
          hi4 = lds_u128(xs + 32 * unit + 16);
          uoff[u] = 256u * u;
        }
        xa[u][0] = lo4.x; xa[u][1] = lo4.y; xa[u][2] = lo4.z; xa[u][3] = lo4.w;
        xa[u][4] = hi4.x; xa[u][5] = hi4.y; xa[u][6] = hi4.z; xa[u][7] = hi4.w;
      }
      const int upt = (units + 31) / 32;       // units per lane this call needs
      const bool full = units == 32 * upt;     // every lane has all of them
      // (xs is rewritten by the next call only after the end-of-call barrier below)

      // ---- rows, stage by stage
      for (int q = 0; q < rows; q += sr, ++i) {
        const int st = i % kStages;
        if (!mbar_wait(smem_u32(&sm.full[st]), (i / kStages) & 1) || *abort_flag) {
          *abort_flag = 1;
          break;
        }
        const int nr = rows - q < sr ? rows - q : sr;
        const uint32_t sbase = ring + st * kStageBytes;
        float *yq = c.y + r0 + q;
        switch (upt) {
          case 1: stage_rows<1>(sbase, nr, rb, laddr, warp, uoff, full, xa, xtot, cm, yq, lane); break;
          case 2: stage_rows<2>(sbase, nr, rb, laddr, warp, uoff, full, xa, xtot, cm, yq, lane); break;
          case 3: stage_rows<3>(sbase, nr, rb, laddr, warp, uoff, full, xa, xtot, cm, yq, lane); break;
          case 4: stage_rows<4>(sbase, nr, rb, laddr, warp, uoff, full, xa, xtot, cm, yq, lane); break;
          case 5: stage_rows<5>(sbase, nr, rb, laddr, warp, uoff, full, xa, xtot, cm, yq, lane); break;
          case 6: stage_rows<6>(sbase, nr, rb, laddr, warp, uoff, full, xa, xtot, cm, yq, lane); break;
          case 7: stage_rows<7>(sbase, nr, rb, laddr, warp, uoff, full, xa, xtot, cm, yq, lane); break;
          default: stage_rows<8>(sbase, nr, rb, laddr, warp, uoff, full, xa, xtot, cm, yq, lane); break;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&sm.empty[st]));
      }
    }

    // ---- this block is done with call ci: the block barrier orders every
    // warp's y stores before thread 0's release (cumulative), which the other
    // blocks acquire before reading.  (One arrival per warp instead measured
    // slower: eight times the atomics on one counter.)
    named_bar(1, kC);
    if (tid == 0) red_release_add(p.bar, 1u);
  }
}

}  // namespace chain
}  // namespace bl
