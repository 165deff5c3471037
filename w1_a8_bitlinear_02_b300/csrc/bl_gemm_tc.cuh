// Tensor-core BitLinear contraction for M > 8 tokens (batched decode and
// prefill), tcgen05 on sm_103a.
//
// sm_103a has no integer MMA (ptxas rejects tcgen05.mma kind::i8 for this
// target), so the int8 x ternary product runs as kind::f16 with bf16
// operands: every code (-1, 0, +1) and every activation code (-128..127) is
// an exact bf16, each product is exact and every partial sum is an integer
// below 127 * K <= 2^24, which fp32 accumulation represents exactly.  The
// accumulator is therefore the exact int32 dot product.
//
// Tile: 128 weight rows (the MMA's M) x BN tokens (the MMA's N) x 64 k per
// pipeline stage.  Roles (320 threads):
//   warp 0      TMA producer: the packed 2-bit weight tile (128 rows x 16 B)
//               and the bf16 activation tile (BN rows x 128 B, 128-byte
//               swizzle) of each stage, completion on one mbarrier.
//   warp 1      allocates TMEM; one lane issues the MMAs (4 x K=16 per stage,
//               A from tensor memory, B from shared memory) and commits each
//               stage back to the producer.
//   warps 2..9  unpack, two groups of four taking alternate stages (so one
//               stage's load-convert-store latency overlaps the next's): warp
//               w expands, for the 32 weight rows of TMEM lane quarter w % 4,
//               each row's 16 packed bytes (64 weights) into bf16 and stores
//               them straight into the stage's A buffer in tensor memory
//               ("pack-store-load-unpack-compute":
//               packed in HBM, unpacked on chip -- "微软AI大模型炸场：0.4GB，
//               CPU就能跑", blog.csdn.net/2401_84494441, section 3, GPU
//               bullet).  Shared memory then only holds the activation and
//               packed tiles, so more stages fit and the A operand costs no
//               shared-memory bandwidth.  Then the epilogue:
//               TMEM -> registers -> y = fl32(acc * c_m), c_m = gamma / s_m.
// Tensor memory: D (accumulator) in columns [0, max(32, BN)), then one
// 32-column A buffer (128 rows x 64 bf16) per stage.
// Split-K (for small tile counts): partial int32 sums are added atomically
// into a workspace zeroed by the preceding activation kernel; the last CTA
// of each tile (an atomic ticket, no spinning) applies the rescale.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cstdint>

#include "bl_pack_quant.cuh"
#include "bl_ptx.cuh"

namespace bl {
namespace tc {

constexpr int kThreads = 320;
constexpr int kUnpackWarps = 8;
constexpr int kUnpackThreads = kUnpackWarps * 32;
constexpr int kBM = 128;                 // weight rows per tile
constexpr int kBK = 64;                  // k per stage
constexpr int kPBytes = kBM * kBK / 4;   // packed weights per stage
constexpr int kSmemBudget = 210 * 1024;
// Token tiles of up to 64 use half the tensor memory (256 columns) and at
// least 80 KB of shared memory, so two blocks share an SM (never three): at a
// few tokens one block's barrier round trips and single-thread MMA issue leave
// the SM mostly idle, and a second block fills it.
__host__ __device__ constexpr int blocks_per_sm(int bn) { return bn <= 64 ? 2 : 1; }

template <int BN>
struct Cfg {
  static constexpr int kBBytes = BN * kBK * 2;
  static constexpr int kStageBytes = kBBytes + kPBytes;
  static constexpr int kDCols = BN < 32 ? 32 : BN;
  static constexpr int kTmemCols = blocks_per_sm(BN) == 2 ? 256 : 512;
  static constexpr int kBySmem = kSmemBudget / kStageBytes;
  static constexpr int kByTmem = (kTmemCols - kDCols) / 32;
  static constexpr int kMin = kBySmem < kByTmem ? kBySmem : kByTmem;
  // even, so each ring slot always serves the same unpack group
  static constexpr int kStages = (kMin < 8 ? kMin : 8) & ~1;
  // stages + up to 1023 bytes of alignment slack + the barrier block
  static constexpr int kSmemRaw = kStages * kStageBytes + 1024 + 3072;
  static constexpr int kSmemBytes = blocks_per_sm(BN) == 2 && kSmemRaw < 80 * 1024 ? 80 * 1024 : kSmemRaw;
  static_assert(BN % 16 == 0 && BN >= 16 && BN <= 256, "MMA N for M = 128");
  static_assert(kStages >= 2, "pipeline depth");
  static_assert(kDCols + 32 * kStages <= kTmemCols, "tensor memory columns");
};

struct Params {
  int N, M;
  int num_kt;        // k tiles in the padded K (Kp / 64)
  int kt_per_split;
  int splits;
  // Stream-K (one split, a persistent grid of one block per SM): block b takes
  // the flattened (output tile, k tile) units [b * units_per, (b + 1) *
  // units_per) ∩ [0, units); tile t is (m tile t / tiles_n, n tile t % tiles_n).
  int streamk;
  int tiles_n;
  int units, units_per;
  const float *gamma;
  const float *scale;  // [M] activation scales (float output only)
  OutSpec out;         // y [M, N]
  int32_t *acc_out;    // [M, N] (int32 output)
  int32_t *ws_acc;     // [M, N] split-K partial sums (float output, splits > 1)
  unsigned *ws_cnt;    // per output tile tickets (float output, splits > 1)
  int32_t *ws_part;    // stream-K: [grid][BN][128] int32 partial tile of each block's first segment
  unsigned *ws_flag;   // stream-K: [grid] set to 1 once that partial is written (zeroed by the
                       // previous kernel on the stream)
};

// A run of k tiles of one output tile and what its epilogue does with it.
enum SegKind {
  kSegFull = 0,   // the whole K: write y
  kSegSplit = 1,  // split-K part: add int32 into ws_acc; the last of the tile's parts writes y
  kSegTail = 2,   // stream-K, first segment of a block, k0 > 0: int32 partial to ws_part[block]
  kSegHead = 3    // stream-K, last segment of a block, k from 0: add ws_part[block + 1], write y
};
struct Seg {
  int n0, m0, k0, nk, kind;
};

// Walks this block's segments in order (one for the plain and split-K grids).
template <int BN>
struct SegWalk {
  int u, u1;
  __device__ __forceinline__ explicit SegWalk(const Params &p) {
    if (p.streamk) {
      u = blockIdx.x * p.units_per;
      u1 = u + p.units_per < p.units ? u + p.units_per : p.units;
    } else {
      u = 0;
      u1 = 1;
    }
  }
  __device__ __forceinline__ bool next(const Params &p, Seg &sg) {
    if (u >= u1) return false;
    if (p.streamk) {
      const int t = u / p.num_kt;
      sg.k0 = u - t * p.num_kt;
      sg.nk = p.num_kt - sg.k0 < u1 - u ? p.num_kt - sg.k0 : u1 - u;
      sg.n0 = (t % p.tiles_n) * kBM;
      sg.m0 = (t / p.tiles_n) * BN;
      sg.kind = (sg.k0 == 0 && sg.nk == p.num_kt) ? kSegFull : (sg.k0 > 0 ? kSegTail : kSegHead);
      u += sg.nk;
    } else {
      sg.n0 = blockIdx.x * kBM;
      sg.m0 = blockIdx.y * BN;
      sg.k0 = blockIdx.z * p.kt_per_split;
      sg.nk = p.num_kt - sg.k0 < p.kt_per_split ? p.num_kt - sg.k0 : p.kt_per_split;
      sg.kind = p.splits == 1 ? kSegFull : kSegSplit;
      u = u1;
    }
    return true;
  }
};

struct Bars {
  uint64_t full[8];
  uint64_t afull[8];
  uint64_t empty[8];
  uint64_t dfull;   // a segment's MMAs are done (phase per segment)
  uint64_t dempty;  // the epilogue has read the accumulator (phase per segment)
  uint32_t tmem_base;
  int abort_flag;
  int last_flag;
  float cscale[256];  // per-token output scale gamma / s_m of this tile
};

// bf16 bytes of (code - 1) for code 0, 1, 2: -1.0 = 0xBF80, 0, +1.0 = 0x3F80.
constexpr uint32_t kTabHi = 0x003F00BFu;
constexpr uint32_t kTabLo = 0x00800080u;

// Four 2-bit codes, one per byte, -> two 32-bit words of bf16 pairs.
__device__ __forceinline__ void codes4_to_bf16(uint32_t codes, uint32_t &w01, uint32_t &w23) {
  const uint32_t t = codes * 0x11u + 0x04040404u;  // selector nibbles [c+4, c] per code
  w01 = __byte_perm(kTabHi, kTabLo, t);
  w23 = __byte_perm(kTabHi, kTabLo, t >> 16);
}

__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned *p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release_u32(unsigned *p, unsigned v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// GROUPED: weights with one scale per group of output rows (the output scale
// is fl32(gamma_g / s_m) per element); a separate instantiation so that the
// per-tensor epilogue stays as tight as before.
template <int BN, bool OUT_I32, bool GROUPED = false>
__global__ void __launch_bounds__(kThreads, blocks_per_sm(BN))
    tc_gemm_kernel(const __grid_constant__ CUtensorMap map_x, const __grid_constant__ CUtensorMap map_w,
                   const Params p) {
  using C = Cfg<BN>;
  constexpr int S = C::kStages;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  const uint32_t b_base = base;
  const uint32_t p_base = b_base + S * C::kBBytes;
  Bars &bars = *reinterpret_cast<Bars *>(smem_raw + (base - raw) + S * C::kStageBytes);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(smem_u32(&bars.full[s]), 1);
      mbar_init(smem_u32(&bars.afull[s]), kUnpackThreads / 2);
      mbar_init(smem_u32(&bars.empty[s]), 1);
    }
    mbar_init(smem_u32(&bars.dfull), 1);
    mbar_init(smem_u32(&bars.dempty), kUnpackThreads);
    bars.abort_flag = 0;
    bars.last_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tensormap(&map_x);
    prefetch_tensormap(&map_w);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&bars.tmem_base), C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars.tmem_base;
  pdl_launch_dependents();
  volatile int *abort_flag = &bars.abort_flag;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      const uint64_t pol_w = policy_evict_first();
      const uint64_t pol_x = policy_evict_last();
      constexpr uint32_t kTx = kPBytes + C::kBBytes;
      // Weights are static inputs: request the first S stages' before the
      // previous kernel ends, their activation tiles after.
      {
        SegWalk<BN> w(p);
        Seg sg;
        int i = 0;
        while (i < S && w.next(p, sg))
          for (int t = 0; t < sg.nk && i < S; ++t, ++i) {
            const uint32_t fb = smem_u32(&bars.full[i]);
            mbar_arrive_expect_tx(fb, kTx);
            tma_load_2d(p_base + i * kPBytes, &map_w, (sg.k0 + t) * 16, sg.n0, fb, pol_w);
          }
      }
      pdl_wait_primary();
      SegWalk<BN> w(p);
      Seg sg;
      int i = 0, issued = 0;
      bool go = true;
      while (go && w.next(p, sg)) {
        for (int t = 0; t < sg.nk; ++t, ++i) {
          const int s = i % S;
          const uint32_t fb = smem_u32(&bars.full[s]);
          if (i >= S) {
            if (!mbar_wait(smem_u32(&bars.empty[s]), ((i / S) - 1) & 1) || *abort_flag) {
              *abort_flag = 1;
              go = false;
              break;
            }
            mbar_arrive_expect_tx(fb, kTx);
            tma_load_2d(p_base + s * kPBytes, &map_w, (sg.k0 + t) * 16, sg.n0, fb, pol_w);
          }
          tma_load_2d(b_base + s * C::kBBytes, &map_x, (sg.k0 + t) * kBK, sg.m0, fb, pol_x);
          issued = i + 1;
        }
      }
      for (int j = issued - S < 0 ? 0 : issued - S; j < issued; ++j)
        mbar_wait(smem_u32(&bars.full[j % S]), (j / S) & 1);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(kBM, BN);
      // afull implies full: the unpack warps arrive only after waiting for a
      // stage's TMA bytes (activation tile included), and mbarrier
      // release/acquire chains are transitive.  (Moving this wait between a
      // stage's MMAs, to overlap it with them, measured slower.)
      SegWalk<BN> w(p);
      Seg sg;
      int i = 0, j = 0;
      bool go = true;
      while (go && w.next(p, sg)) {
        // the accumulator is reused: the previous segment's epilogue must have read it
        if (j > 0 && !mbar_wait(smem_u32(&bars.dempty), (j - 1) & 1)) {
          *abort_flag = 1;
          break;
        }
        tc_fence_after();
        for (int t = 0; t < sg.nk; ++t, ++i) {
          const int s = i % S;
          if (!mbar_wait(smem_u32(&bars.afull[s]), (i / S) & 1)) {
            *abort_flag = 1;
            go = false;
            break;
          }
          tc_fence_after();
          const uint32_t at = tmem + C::kDCols + 32u * s;
          const uint64_t bd = smem_desc_sw128(b_base + s * C::kBBytes);
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk)
            mma_bf16_ts(tmem, at + 8u * kk, bd + 2u * kk, idesc, (t | kk) != 0 ? 1u : 0u);
          mma_commit(smem_u32(&bars.empty[s]));
        }
        mma_commit(smem_u32(&bars.dfull));  // fires once the segment's MMAs are done
        ++j;
      }
    }
  } else {
    // ------------------------------------------------------------ unpack + epilogue
    const int u = tid - 64;            // 0 .. 255
    const int q = warp & 3;            // TMEM lane quarter this warp may access
    const int h = (warp - 2) >> 2;     // unpack group: stages i = h (mod 2)
    const int row = 32 * q + lane;     // weight row of the tile
    const uint32_t lane_off = static_cast<uint32_t>(32 * q) << 16;
    SegWalk<BN> w(p);
    Seg sg;
    int i = 0, j = 0;
    bool alive = true;
    while (w.next(p, sg)) {
      for (int t = 0; t < sg.nk; ++t, ++i) {
        if ((i & 1) != h || !alive) continue;
        const int s = i % S;
        if (!mbar_wait(smem_u32(&bars.full[s]), (i / S) & 1) || *abort_flag) {
          *abort_flag = 1;
          alive = false;
          continue;
        }
        const uint4 wv = lds_u128(p_base + s * kPBytes + row * 16);
        const uint32_t words[4] = {wv.x, wv.y, wv.z, wv.w};
        uint32_t v[32];
#pragma unroll
        for (int wi = 0; wi < 4; ++wi) {
#pragma unroll
          for (int i4 = 0; i4 < 4; ++i4)  // k = 16 wi + 4 i4 .. +3
            codes4_to_bf16((words[wi] >> (2 * i4)) & 0x03030303u, v[8 * wi + 2 * i4], v[8 * wi + 2 * i4 + 1]);
        }
        tmem_st_32x32b_x32(tmem + lane_off + C::kDCols + 32u * s, v);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(smem_u32(&bars.afull[s]));
      }

      // -------------------------------------------------------- epilogue of this segment
      // scale / workspaces come from the previous kernel on the stream
      pdl_wait_primary();
      // every epilogue thread is past the previous segment's epilogue (which
      // reads cscale) before it is rewritten
      named_bar(5, kUnpackThreads);
      if constexpr (!OUT_I32) {
        const float g = *p.gamma;
        for (int c = u; c < BN; c += kUnpackThreads)
          bars.cscale[c] = (sg.m0 + c < p.M) ? __fdiv_rn(g, p.scale[sg.m0 + c]) : 0.0f;
      }
      bool ok = alive && mbar_wait(smem_u32(&bars.dfull), j & 1);
      // One decision for all epilogue warps (they share named barriers and
      // warp-collective TMEM loads below); also orders the cscale writes.
      ok = !named_bar_or(4, kUnpackThreads, !ok || *abort_flag);
      tc_fence_after();
      const int n = sg.n0 + row;
      const int m0 = sg.m0;
      if (ok && sg.kind == kSegHead) {
        // the rest of this tile's K is the next block's first segment
        bool late = false;
        if (u == 0) {
          const long long t0 = clock64();
          while (ld_acquire_u32(p.ws_flag + blockIdx.x + 1) == 0u) {
            if (clock64() - t0 > kWaitLimitCycles) {
              atomicOr(&g_dev_error, kDevErrTimeout);
              late = true;
              break;
            }
          }
        }
        ok = !named_bar_or(4, kUnpackThreads, late);
      }
      if (ok) {
        const int32_t *part_in = p.ws_part + static_cast<int64_t>(blockIdx.x + 1) * BN * kBM;
        int32_t *part_out = p.ws_part + static_cast<int64_t>(blockIdx.x) * BN * kBM;
        const int kind = sg.kind;
        // one loop per kind: the accumulator columns c0 .. c0 + 31 of row n
#pragma unroll 1
        for (int c0 = 32 * h; c0 < BN; c0 += 64) {
          uint32_t r[32];
          tmem_ld_32x32b_x32(tmem + lane_off + c0, r);
          tmem_ld_wait();
          // below 32 tokens a tile has BN < 32 accumulator columns: the rest
          // of the 32 loaded are not this tile's (and the partial tile in the
          // workspace has BN rows)
          constexpr int kCols = BN < 32 ? BN : 32;
          if (kind == kSegTail) {
#pragma unroll
            for (int jj = 0; jj < kCols; ++jj)
              part_out[(c0 + jj) * kBM + row] = static_cast<int>(__uint_as_float(r[jj]));
          } else if (kind == kSegSplit) {
            if (n < p.N) {
#pragma unroll
              for (int jj = 0; jj < kCols; ++jj) {
                const int m = m0 + c0 + jj;
                if (m < p.M) {
                  const int64_t o = static_cast<int64_t>(m) * p.N + n;
                  if constexpr (OUT_I32)
                    atomicAdd(&p.acc_out[o], static_cast<int>(__uint_as_float(r[jj])));
                  else
                    atomicAdd(&p.ws_acc[o], static_cast<int>(__uint_as_float(r[jj])));
                }
              }
            }
          } else {
            if (kind == kSegHead) {
#pragma unroll
              for (int jj = 0; jj < kCols; ++jj)
                r[jj] = __float_as_uint(static_cast<float>(static_cast<int>(__uint_as_float(r[jj])) +
                                                           __ldcg(part_in + (c0 + jj) * kBM + row)));
            }
            if (n < p.N) {
#pragma unroll
              for (int jj = 0; jj < kCols; ++jj) {
                const int m = m0 + c0 + jj;
                if (m < p.M) {
                  const int64_t o = static_cast<int64_t>(m) * p.N + n;
                  const int v = static_cast<int>(__uint_as_float(r[jj]));
                  if constexpr (OUT_I32) {
                    p.acc_out[o] = v;
                  } else {
                    float cmn;
                    if constexpr (GROUPED)
                      cmn = group_scale(p.out, n, __ldg(p.scale + m));
                    else
                      cmn = bars.cscale[c0 + jj];
                    put_y(p.out, o, __fmul_rn(static_cast<float>(v), cmn));
                  }
                }
              }
            }
          }
        }
        if (sg.kind == kSegTail) {
          // publish this block's partial for the block that owns the tile
          __threadfence();
          named_bar(3, kUnpackThreads);
          if (u == 0) st_release_u32(p.ws_flag + blockIdx.x, 1u);
        }
        if constexpr (!OUT_I32) {
          if (sg.kind == kSegSplit) {
            __threadfence();
            named_bar(3, kUnpackThreads);
            if (u == 0) {
              const unsigned t = atomicAdd(&p.ws_cnt[blockIdx.y * gridDim.x + blockIdx.x], 1u);
              bars.last_flag = (t == static_cast<unsigned>(p.splits - 1)) ? 1 : 0;
            }
            named_bar(3, kUnpackThreads);
            if (bars.last_flag) {
              __threadfence();
              if (n < p.N) {
                for (int c = h; c < BN; c += 2) {
                  const int m = m0 + c;
                  if (m >= p.M) break;
                  const int64_t o = static_cast<int64_t>(m) * p.N + n;
                  const int v = __ldcg(&p.ws_acc[o]);
                  float cmn;
                  if constexpr (GROUPED)
                    cmn = group_scale(p.out, n, __ldg(p.scale + m));
                  else
                    cmn = bars.cscale[c];
                  put_y(p.out, o, __fmul_rn(static_cast<float>(v), cmn));
                }
              }
            }
          }
        }
      }
      tc_fence_before();
      mbar_arrive(smem_u32(&bars.dempty));  // the accumulator may be overwritten
      ++j;
    }
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

}  // namespace tc
}  // namespace bl
