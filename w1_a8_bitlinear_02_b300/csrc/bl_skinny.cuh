// Tensor-core BitLinear forward for a few tokens (3 <= M <= 64, batched
// decode), tcgen05 on sm_103a: one launch per call, no workspace.
//
// At a few tokens one MMA instruction (128 weight rows x 16..64 tokens x 16 k)
// is little work: the issue latency of one issuing thread (about 45 cycles per
// instruction on B300, plus about 100 for each barrier wait and 60 for each
// commit) bounds the rate, not the tensor pipe.  So the k tiles go in stages
// of four (16 MMAs per barrier wait) and NI issuing warps, each with an
// accumulator of its own, take the stages in turn.  Stage t belongs to lane
// t mod NI: one issuer, one group of four unpack warps (one per tensor-memory
// lane quarter) and one tensor-memory A slot, so every barrier between them
// alternates strictly between one waiter and one signaller (a parity wait can
// never be two phases behind).  The weight ring depth is a multiple of NI for
// the same reason.  The packed weights are the bytes that matter; the rest is
// arranged around their stream and around the latency of one call:
//   * K is split over a thread-block cluster of CS blocks that share one
//     128-row tile; each block owns a contiguous run of 64-k tiles.
//   * Weights are static, so their first stages are loaded by TMA and
//     expanded to bf16 in tensor memory (the A operand) before the kernel
//     waits for the previous one on the stream.
//   * The activations are quantised here, per token to int8 absmax ("20亿参数
//     仅0.4GB…「原生1.58bit」大模型", blog.csdn.net/soaring_casia, section 2
//     "BitLinear层", item 2).  bf16 rows arrive by TMA straight into the MMA's
//     B operand layout (128-byte swizzle, K-major, zero outside M x K); each
//     block sends its partial per-token absmax to the others' shared memory,
//     and the integer codes overwrite the values in place.  Other inputs (f32,
//     int8 codes, unaligned rows) are read with plain loads.
//   * Each block sends its partial sums of the tokens m = r (mod CS) to block
//     r's shared memory; after one cluster barrier (no block touches another's
//     shared memory past it, so none can exit while it is still written)
//     block r adds them and writes y = fl32(acc * c_m), c_m = fl32(gamma / s_m).
// Exactness as in the tensor-core GEMM: bf16 codes, fp32 accumulation of
// integers below 2^24.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cstdint>
#include <type_traits>

#include "bl_gemm_tc.cuh"
#include "bl_pack_quant.cuh"
#include "bl_ptx.cuh"

namespace bl {
namespace sk {

constexpr int kBM = 128;                // weight rows per tile
constexpr int kBK = 64;                 // k per tile
constexpr int kKT = 4;                  // k tiles per stage
constexpr int kTile = kBM * kBK / 4;    // packed bytes per k tile
constexpr int kStage = kKT * kTile;     // packed bytes per stage
constexpr int kMaxWS = 16;              // weight ring stages, at most
constexpr int kMaxNI = 3;
constexpr int kTmemCols = 512;
constexpr int kMaxM = 64;
constexpr int kMaxCS = 8;

// Activation source.
constexpr int kXF32 = 0;
constexpr int kXBF16 = 1;
constexpr int kXInt8 = 2;

// Lanes (issuer + unpack group + A slot) per token tile: three up to 32
// tokens, two at 64 (the accumulators then take 128 columns).
__host__ __device__ constexpr int lanes_for(int bn) { return bn <= 32 ? 3 : 2; }

template <int BN>
struct Cfg {
  static constexpr int kNI = lanes_for(BN);      // issuers = unpack groups = A slots
  static constexpr int kUW = 4 * kNI;            // unpack warps
  static constexpr int kU0 = 1 + kNI;            // first unpack warp
  static constexpr int kWarps = 1 + kNI + kUW;   // producer, issuers, unpack
  static constexpr int kThreads = 32 * kWarps;
  static constexpr int kDC = BN < 32 ? 32 : BN;  // tensor-memory columns per accumulator
  static constexpr int kACol = kNI * kDC;        // first column of the A slots
  static constexpr int kAtom = BN * 128;         // B operand bytes per k tile
  static_assert(BN == 16 || BN == 32 || BN == 64, "token tile");
  static_assert(kNI <= kMaxNI, "lanes");
  static_assert(kACol + kNI * 32 * kKT <= kTmemCols, "tensor memory columns");
};

struct Bars {
  uint64_t wfull[kMaxWS], wempty[kMaxWS];
  uint64_t afull[kMaxNI], afree[kMaxNI];
  uint64_t dfull, xfull, xbar;
  uint32_t tmem_base;
  int abort_flag;
  float amax[kMaxM];             // this block's absmax per token over its k range
  float amax_all[kMaxCS][kMaxM]; // every block's, sent by the blocks themselves
  float sc[kMaxM];               // s_m = 127 / max(absmax, 1e-5)
  float cscale[kMaxM];           // gamma / s_m
};
static_assert(sizeof(Bars) <= 4096, "barrier block");

struct Params {
  const void *x;        // [M, K]: f32 / bf16 activations, or int8 codes
  const float *scale;   // int8 codes with float output: their scales [M]
  const float *gamma;   // float output
  OutSpec out;          // y [M, N]
  int32_t *acc;         // [M, N] (int32 output)
  int M, N, K;
  int num_kt;           // 64-k tiles in the padded K
  int kt_per;           // k tiles per block (the last block of a cluster may have fewer)
  int cs;               // blocks per cluster (K split)
  int ws;               // weight ring stages (a multiple of the lanes)
  int x_tma;            // bf16 rows come by TMA (map_x valid)
  int act;              // activation before quantisation (kActNone / kActRelu2)
};

// Eight bf16 codes (integers in [-128, 127], exact) as four bf16 pairs.
__device__ __forceinline__ void codes8_bf16(const int (&q)[8], uint32_t (&w)[4]) {
#pragma unroll
  for (int i = 0; i < 4; ++i)
    w[i] = (__float_as_uint(static_cast<float>(q[2 * i])) >> 16) |
           (__float_as_uint(static_cast<float>(q[2 * i + 1])) & 0xFFFF0000u);
}

__device__ __forceinline__ void bf16x8_f32(const uint4 u, float (&v)[8]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    v[2 * j] = __uint_as_float(w[j] << 16);
    v[2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
  }
}

template <int BN, int XM, bool OUT_I32>
__global__ void __launch_bounds__(Cfg<BN>::kThreads, 1)
    skinny_kernel(const __grid_constant__ CUtensorMap map_w, const __grid_constant__ CUtensorMap map_x,
                  const Params p) {
  using C = Cfg<BN>;
  constexpr int NI = C::kNI;
  constexpr int kWarps = C::kWarps;
  constexpr int kThreads = C::kThreads;
  constexpr int kU0 = C::kU0;
  constexpr int kUW = C::kUW;
  using XT = typename std::conditional<XM == kXF32, float, __nv_bfloat16>::type;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  const int cs = p.cs;
  const int ms = (p.M + cs - 1) / cs;  // tokens per finishing block, at most
  const uint32_t b_base = base;
  const uint32_t w_base = b_base + static_cast<uint32_t>(p.kt_per) * C::kAtom;
  const uint32_t red_base = w_base + static_cast<uint32_t>(p.ws) * kStage;  // [cs][ms][128] int32
  const uint32_t bars_off = red_base + (cs > 1 ? static_cast<uint32_t>(cs * ms * kBM * 4) : 0u);
  Bars &bars = *reinterpret_cast<Bars *>(smem_raw + (bars_off - raw));

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = cluster_ctarank();
  const int n0 = blockIdx.y * kBM;
  const int kt0 = static_cast<int>(rank) * p.kt_per;
  int nkt = p.num_kt - kt0;
  if (nkt > p.kt_per) nkt = p.kt_per;  // >= 1: the plan gives every block a k tile
  const int nst = (nkt + kKT - 1) / kKT;  // stages of this block
  const int ws = p.ws;

  // barriers, one per thread
  if (tid < ws) {
    mbar_init(smem_u32(&bars.wfull[tid]), 1);
    mbar_init(smem_u32(&bars.wempty[tid]), 4);
  } else if (tid >= 32 && tid < 32 + NI) {
    mbar_init(smem_u32(&bars.afull[tid - 32]), 4);
    mbar_init(smem_u32(&bars.afree[tid - 32]), 1);
  } else if (tid == 64) {
    mbar_init(smem_u32(&bars.dfull), NI);
    mbar_init(smem_u32(&bars.xfull), 1);
    mbar_init(smem_u32(&bars.xbar), cs > 1 ? cs - 1 : 1);
    bars.abort_flag = 0;
  }
  fence_barrier_init();
  if (warp == 1) {
    tmem_alloc(smem_u32(&bars.tmem_base), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // every block's barriers exist before any block arrives on them remotely
  if (cs > 1) cluster_sync_all();
  const uint32_t tmem = bars.tmem_base;
  pdl_launch_dependents();
  volatile int *abort_flag = &bars.abort_flag;

  // Weights are static inputs: request the first stages before the previous
  // kernel on the stream has finished.
  int issued = 0;
  uint64_t pol_w = 0;
  if (tid == 0) {
    pol_w = policy_evict_first();
    prefetch_tensormap(&map_w);
    if (p.x_tma) prefetch_tensormap(&map_x);
    const int pre = nst < ws ? nst : ws;
    for (int st = 0; st < pre; ++st) {
      const int nk = nkt - st * kKT < kKT ? nkt - st * kKT : kKT;
      const uint32_t fb = smem_u32(&bars.wfull[st]);
      mbar_arrive_expect_tx(fb, nk * kTile);
      for (int i = 0; i < nk; ++i)
        tma_load_2d(w_base + st * kStage + i * kTile, &map_w, (kt0 + st * kKT + i) * 16, n0, fb, pol_w);
    }
    issued = pre;
  }

  // one stage of weights -> bf16 in tensor memory (unpack warps)
  const int ug = (warp - kU0) >> 2;  // unpack group = lane (warps of other roles: unused)
  const int q = warp & 3;            // the TMEM lane quarter this warp may access
  const int row = 32 * q + lane;
  const uint32_t lane_off = static_cast<uint32_t>(32 * q) << 16;
  auto unpack_stage = [&](int st) -> bool {
    const int s = st % ws;
    if (!mbar_wait(smem_u32(&bars.wfull[s]), (st / ws) & 1) || *abort_flag) return false;
    const int a = st % NI;
    if (st >= NI && !mbar_wait(smem_u32(&bars.afree[a]), ((st / NI) - 1) & 1)) return false;
    tc_fence_after();
    const int nk = nkt - st * kKT < kKT ? nkt - st * kKT : kKT;
    for (int i = 0; i < nk; ++i) {
      const uint4 wv = lds_u128(w_base + s * kStage + i * kTile + row * 16);
      const uint32_t words[4] = {wv.x, wv.y, wv.z, wv.w};
      uint32_t v[32];
#pragma unroll
      for (int wi = 0; wi < 4; ++wi)
#pragma unroll
        for (int i4 = 0; i4 < 4; ++i4)  // k = 16 wi + 4 i4 .. +3
          tc::codes4_to_bf16((words[wi] >> (2 * i4)) & 0x03030303u, v[8 * wi + 2 * i4],
                             v[8 * wi + 2 * i4 + 1]);
      tmem_st_32x32b_x32(tmem + lane_off + C::kACol + 32u * (kKT * a + i), v);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&bars.wempty[s]));
    tmem_st_wait();
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&bars.afull[a]));
    return true;
  };
  const bool is_unpack = warp >= kU0;
  if (is_unpack && ug < nst && !unpack_stage(ug)) *abort_flag = 1;

  pdl_wait_primary();  // x (and the scales) come from the previous kernel

  // ---------------------------------------------------------------- activations
  const int kbeg = kt0 * kBK;
  int kend = (kt0 + nkt) * kBK;
  if (kend > p.K) kend = p.K;
  const int cpr = nkt * 8;  // 8-element (16-byte) chunks per token row of the B operand
  // chunk r of token m: k tile r / 8, 16-byte chunk (r % 8) ^ (m % 8) of row m
  auto b_chunk = [&](int m, int r) -> uint32_t {
    return b_base + (r >> 3) * C::kAtom + m * 128 + (((r & 7) ^ (m & 7)) << 4);
  };
  if constexpr (XM == kXBF16) {
    if (p.x_tma) {
      if (tid == 0) {
        const uint32_t xb = smem_u32(&bars.xfull);
        mbar_arrive_expect_tx(xb, nkt * C::kAtom);
        for (int j = 0; j < nkt; ++j)
          tma_load_2d(b_base + j * C::kAtom, &map_x, (kt0 + j) * kBK, 0, xb, policy_evict_last());
      }
      if (!mbar_wait(smem_u32(&bars.xfull), 0)) *abort_flag = 1;
      // absmax per token from shared memory (zeros outside M x K)
      for (int m = warp; m < p.M; m += kWarps) {
        float a = 0.0f;
        for (int r = lane; r < cpr; r += 32) {
          float v[8];
          bf16x8_f32(lds_u128(b_chunk(m, r)), v);
#pragma unroll
          for (int i = 0; i < 8; ++i) a = fmaxf(a, fabsf(p.act == kActRelu2 ? relu2f(v[i]) : v[i]));
        }
        a = warp_max_nonneg(a);
        if (lane == 0) bars.amax[m] = a;
      }
    }
  }
  if constexpr (XM != kXInt8) {
    if (XM != kXBF16 || !p.x_tma) {
      const XT *x = static_cast<const XT *>(p.x);
      const bool vec = (p.K % 8 == 0) && al16(x);
      for (int m = warp; m < p.M; m += kWarps) {
        const XT *xr = x + static_cast<int64_t>(m) * p.K;
        float a = 0.0f;
        if (vec) {
#pragma unroll 4
          for (int k = kbeg + 8 * lane; k < kend; k += 256) {
            float v[8];
            load8(xr + k, v);
#pragma unroll
            for (int i = 0; i < 8; ++i) a = fmaxf(a, fabsf(p.act == kActRelu2 ? relu2f(v[i]) : v[i]));
          }
        } else {
#pragma unroll 4
          for (int k = kbeg + lane; k < kend; k += 32) {
            const float v = to_f32(xr[k]);
            a = fmaxf(a, fabsf(p.act == kActRelu2 ? relu2f(v) : v));
          }
        }
        a = warp_max_nonneg(a);
        if (lane == 0) bars.amax[m] = a;
      }
    }
    __syncthreads();
    if (cs > 1) {
      // send this block's absmax to every other block of the cluster
      if (tid < p.M) {
        const float a = bars.amax[tid];
        bars.amax_all[rank][tid] = a;
        const uint32_t la = smem_u32(&bars.amax_all[rank][tid]);
        for (int r = 0; r < cs; ++r)
          if (r != static_cast<int>(rank)) st_dsmem_u32(dsmem_map(la, r), __float_as_uint(a));
        fence_cluster();
      }
      __syncthreads();
      if (tid == 0)
        for (int r = 0; r < cs; ++r)
          if (r != static_cast<int>(rank)) mbar_arrive_remote(dsmem_map(smem_u32(&bars.xbar), r));
    }
  }
  if (tid < p.M) {
    float s;
    if constexpr (XM != kXInt8) {
      float a = bars.amax[tid];
      if (cs > 1) {
        if (!mbar_wait_cluster(smem_u32(&bars.xbar), 0)) *abort_flag = 1;
        for (int r = 0; r < cs; ++r) a = fmaxf(a, bars.amax_all[r][tid]);
      }
      s = act_scale(a);
    } else {
      s = OUT_I32 ? 1.0f : p.scale[tid];
    }
    bars.sc[tid] = s;
    bars.cscale[tid] = OUT_I32 ? 0.0f : __fdiv_rn(*p.gamma, s);
  }
  __syncthreads();
  {
    const int total = BN * cpr;
    if (XM == kXBF16 && p.x_tma) {
      // codes overwrite the values in place (rows m >= M are zero already)
      for (int c = tid; c < p.M * cpr; c += kThreads) {
        const int m = c / cpr;
        const int r = c - m * cpr;
        const uint32_t ad = b_chunk(m, r);
        float v[8];
        bf16x8_f32(lds_u128(ad), v);
        const float s = bars.sc[m];
        int qv[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) qv[i] = quant_one(p.act == kActRelu2 ? relu2f(v[i]) : v[i], s);
        uint32_t w[4];
        codes8_bf16(qv, w);
        sts_u128(ad, w[0], w[1], w[2], w[3]);
      }
    } else {
      bool vec;
      if constexpr (XM == kXInt8)
        vec = (p.K % 8 == 0) && ((reinterpret_cast<uintptr_t>(p.x) & 7u) == 0);
      else
        vec = (p.K % 8 == 0) && al16(p.x);
      for (int c = tid; c < total; c += kThreads) {
        const int m = c / cpr;
        const int r = c - m * cpr;
        const int k = kbeg + 8 * r;
        uint32_t w[4] = {0u, 0u, 0u, 0u};
        if (m < p.M && k < p.K) {
          int qv[8];
          if constexpr (XM == kXInt8) {
            const int8_t *xr = static_cast<const int8_t *>(p.x) + static_cast<int64_t>(m) * p.K;
            if (vec && k + 8 <= p.K) {
              const uint2 u = *reinterpret_cast<const uint2 *>(xr + k);
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                qv[i] = static_cast<int8_t>((u.x >> (8 * i)) & 0xFFu);
                qv[i + 4] = static_cast<int8_t>((u.y >> (8 * i)) & 0xFFu);
              }
            } else {
#pragma unroll
              for (int i = 0; i < 8; ++i) qv[i] = (k + i < p.K) ? xr[k + i] : 0;
            }
          } else {
            const XT *xr = static_cast<const XT *>(p.x) + static_cast<int64_t>(m) * p.K;
            float v[8];
            if (vec && k + 8 <= p.K) {
              load8(xr + k, v);
            } else {
#pragma unroll
              for (int i = 0; i < 8; ++i) v[i] = (k + i < p.K) ? to_f32(xr[k + i]) : 0.0f;
            }
            const float s = bars.sc[m];
#pragma unroll
            for (int i = 0; i < 8; ++i) qv[i] = quant_one(p.act == kActRelu2 ? relu2f(v[i]) : v[i], s);
          }
          codes8_bf16(qv, w);
        }
        sts_u128(b_chunk(m, r), w[0], w[1], w[2], w[3]);
      }
    }
  }
  fence_proxy_async_smem();  // generic-proxy writes, read by the tensor core
  __syncthreads();

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      for (int st = issued; st < nst; ++st) {
        const int s = st % ws;
        if (!mbar_wait(smem_u32(&bars.wempty[s]), ((st / ws) - 1) & 1) || *abort_flag) {
          *abort_flag = 1;
          break;
        }
        const int nk = nkt - st * kKT < kKT ? nkt - st * kKT : kKT;
        const uint32_t fb = smem_u32(&bars.wfull[s]);
        mbar_arrive_expect_tx(fb, nk * kTile);
        for (int i = 0; i < nk; ++i)
          tma_load_2d(w_base + s * kStage + i * kTile, &map_w, (kt0 + st * kKT + i) * 16, n0, fb, pol_w);
        issued = st + 1;
      }
      // no copy of this block may still be in flight when it exits
      for (int st = issued - ws < 0 ? 0 : issued - ws; st < issued; ++st)
        mbar_wait(smem_u32(&bars.wfull[st % ws]), (st / ws) & 1);
    }
  } else if (warp <= NI) {
    // ------------------------------------------------------------ MMA issuers
    const int j = warp - 1;
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(kBM, BN);
      const uint32_t d = tmem + static_cast<uint32_t>(j * C::kDC);
      for (int st = j; st < nst; st += NI) {
        const int a = st % NI;  // == j
        if (!mbar_wait(smem_u32(&bars.afull[a]), (st / NI) & 1)) {
          *abort_flag = 1;
          break;
        }
        tc_fence_after();
        const int nk = nkt - st * kKT < kKT ? nkt - st * kKT : kKT;
        for (int i = 0; i < nk; ++i) {
          const uint32_t at = tmem + C::kACol + 32u * (kKT * a + i);
          const uint64_t bd = smem_desc_sw128(b_base + (st * kKT + i) * C::kAtom);
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk)
            mma_bf16_ts(d, at + 8u * kk, bd + 2u * kk, idesc, (st != j || i != 0 || kk != 0) ? 1u : 0u);
        }
        mma_commit(smem_u32(&bars.afree[a]));
      }
      mma_commit(smem_u32(&bars.dfull));  // fires once this issuer's MMAs are done
    }
  } else {
    // ------------------------------------------------------------ unpack
    for (int st = ug + NI; st < nst; st += NI)
      if (!unpack_stage(st)) {
        *abort_flag = 1;
        break;
      }

    // ------------------------------------------------------------ epilogue
    bool ok = mbar_wait(smem_u32(&bars.dfull), 0);
    ok = !named_bar_or(1, kUW * 32, !ok || *abort_flag);
    tc_fence_after();
    const int nd = nst < NI ? nst : NI;
    const int n = n0 + row;
    if (ok) {
      for (int cc = ug; cc < BN / 16; cc += NI) {
        int sum[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) sum[i] = 0;
        for (int j = 0; j < nd; ++j) {
          uint32_t r[16];
          tmem_ld_32x32b_x16(tmem + lane_off + static_cast<uint32_t>(j * C::kDC + 16 * cc), r);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 16; ++i) sum[i] += static_cast<int>(__uint_as_float(r[i]));
        }
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int m = 16 * cc + i;
          if (m >= p.M) break;
          if (cs == 1) {
            if (n < p.N) {
              const int64_t o = static_cast<int64_t>(m) * p.N + n;
              if constexpr (OUT_I32)
                p.acc[o] = sum[i];
              else
                put_y(p.out, o, __fmul_rn(static_cast<float>(sum[i]),
                                          p.out.gvec ? group_scale(p.out, n, bars.sc[m]) : bars.cscale[m]));
            }
          } else {
            // to block m % cs, slot [this block][m / cs][row]
            const int o = m % cs;
            const uint32_t la =
                red_base + static_cast<uint32_t>(((static_cast<int>(rank) * ms + m / cs) * kBM + row) * 4);
            if (o == static_cast<int>(rank))
              asm volatile("st.shared.u32 [%0], %1;" ::"r"(la), "r"(static_cast<uint32_t>(sum[i])) : "memory");
            else
              st_dsmem_u32(dsmem_map(la, o), static_cast<uint32_t>(sum[i]));
          }
        }
      }
    }
    tc_fence_before();
  }

  if (cs > 1) {
    // Every block's partial sums are in place after this barrier, and no
    // block touches another's shared memory past it.
    cluster_sync_all();
    // this block's tokens m = rank (mod cs): add the cs partial sums
    const int nm = (p.M - static_cast<int>(rank) + cs - 1) / cs;
    {
      for (int idx = tid; idx < nm * kBM; idx += kThreads) {
        const int mi = idx / kBM;
        const int r = idx % kBM;
        const int m = static_cast<int>(rank) + cs * mi;
        const int n = n0 + r;
        if (n < p.N) {
          int sum = 0;
          for (int c = 0; c < cs; ++c) sum += static_cast<int>(lds_u32(red_base + ((c * ms + mi) * kBM + r) * 4));
          const int64_t o = static_cast<int64_t>(m) * p.N + n;
          if constexpr (OUT_I32)
            p.acc[o] = sum;
          else
            put_y(p.out, o, __fmul_rn(static_cast<float>(sum),
                                      p.out.gvec ? group_scale(p.out, n, bars.sc[m]) : bars.cscale[m]));
        }
      }
    }
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace sk
}  // namespace bl
