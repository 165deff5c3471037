// Decode chain: a sequence of M = 1 BitLinear forwards in one persistent
// launch.  A call may read an earlier call's output as its input.
//
// A decode step runs the projections of every layer one after another
// ("BitNet b1.58 2B4T" architecture: QKV, O, FFN up, FFN down per layer;
// "20亿参数仅0.4GB…「原生1.58bit」大模型", blog.csdn.net/soaring_casia,
// section 2).  As separate launches each call pays a kernel boundary although
// its packed weights -- static inputs -- are a fraction of a microsecond of
// HBM time.  Here one block per SM stays resident for the whole chain:
//   * its producer thread streams the block's rows of every call, call after
//     call, into one bulk-copy ring: the weights of later calls arrive while
//     earlier calls compute, limited only by the ring's size ("pack-store-
//     load-unpack-compute", 微软AI大模型炸场：0.4GB, blog.csdn.net/2401_84494441,
//     section 3, GPU bullet, carried across calls);
//   * the consumer warps run the calls in order: quantise the input (per-token
//     absmax, once per block into shared memory), then run the block's rows
//     (masked dp4a on the packed codes, exact int32 sums, y = fl32(acc * c),
//     c = fl32(gamma / s)).
// Dependencies between calls come in two forms, both found by the host from
// the calls' buffers:
//   * mailbox: when a call's x lies inside an earlier call's y, that earlier
//     call also writes each output as one 8-byte word {value, tag} into the
//     workspace, and the reader polls those words directly: the tag says the
//     value is there, so no barrier, fence or separate flag is needed (an
//     aligned 64-bit store is seen whole or not at all).  The tag holds the
//     producing call and a per-launch sequence number kept in the workspace,
//     so words left by an earlier launch never match;
//   * grid barrier: any other overlap (an input read from memory that an
//     earlier call wrote, an output that overwrites an earlier input or
//     output) makes every block finish all earlier calls first (one release-add
//     per block on a counter, acquire-spin until all have arrived).
// All blocks must be resident at once (they may wait for each other): the
// launch is cooperative, one block per SM.
#pragma once

#include <cuda_bf16.h>
#include <cstdint>

#include "bl_pack_quant.cuh"
#include "bl_ptx.cuh"

namespace bl {
namespace chain {

constexpr int kMaxCalls = 256;
constexpr int kCW = 16;                   // consumer warps
constexpr int kThreads = (kCW + 1) * 32;  // + one producer warp
constexpr int kC = kCW * 32;              // consumer threads
constexpr int kUPT = 8;                   // 8-byte units per lane: a warp's chunk spans 256 units (8192 weights)
constexpr int kMaxK = 32768;              // longer rows are split over warps (at most 4 per row)
constexpr int kMaxN = 1 << 30;           // row indices stay far inside int
constexpr int kStageBytes = 32 * 1024;
constexpr int kStages = 5;
constexpr int kMaxSplitRows = 8;          // rows per stage when a row is split over warps
constexpr int kJM = 2;                    // x vectors of 8 per consumer thread kept in registers
constexpr int kSmemFixed = 22 * 1024;     // barriers, reductions and the call table
constexpr int kSmemBytes = kSmemFixed + kStages * kStageBytes + kMaxK;  // + activation codes

// Control words at the start of the workspace (bytes 0..255).
constexpr int kCtlBar = 0;    // grid-barrier arrivals of this launch
constexpr int kCtlDone = 1;   // blocks finished with this launch
constexpr int kCtlSeq = 32;   // launches completed on this workspace (tags)
constexpr int kMailboxOffset = 256;

// Call flags.
constexpr int kFlagBf16 = 1;      // x is bf16 (else fp32)
constexpr int kFlagRelu2 = 2;     // quantise relu2(x)
constexpr int kFlagBarrier = 4;   // every block finishes all earlier calls first

struct Call {
  const uint8_t *packed;  // [N, 16 * ceil(K / 64)]
  const float *gamma;
  const void *x;          // [K] f32 or bf16 (read when mb_in is null)
  float *y;               // [N]
  uint64_t *mb_out;       // this call's output words [N] {value bits, tag}, or null
  const uint64_t *mb_in;  // the words holding x [K] (inside an earlier call's mb_out), or null
  int N, K;
  int rpc;                // rows per block
  int flags;
  int split_log2;         // warps per row: 1 << split_log2
  int chunk;              // 8-byte units per warp chunk of a row
  int stage_rows;         // rows per ring stage
  int src;                // the call that wrote mb_in
};
static_assert(sizeof(Call) % 4 == 0, "call table copied in words");

struct Params {
  int n;                  // calls
  unsigned *ctl;          // workspace control words
  Call c[kMaxCalls];
};

struct Smem {
  uint64_t full[kStages];
  uint64_t empty[kStages];
  float fred[kCW];
  int32_t part[kStages][kMaxSplitRows];
  uint32_t cnt[kStages][kMaxSplitRows];
  uint32_t seq_tag;
  int abort_flag;
  Call calls[kMaxCalls];  // the parameters, copied once: indexed reads of the
                          // parameter space go through the constant cache
};
static_assert(sizeof(Smem) <= kSmemFixed, "fixed shared-memory region");

__device__ __forceinline__ void red_release_add(unsigned *p, unsigned v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ unsigned ld_acquire(const unsigned *p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
// One output word {value bits (low half), tag (high half)}: a single aligned
// 64-bit store, so a reader sees both halves or neither.
__device__ __forceinline__ void st_word(uint64_t *p, float v, uint32_t tag) {
  const uint64_t w = (static_cast<uint64_t>(tag) << 32) | __float_as_uint(v);
  asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" ::"l"(p), "l"(w) : "memory");
}
// Two consecutive output words (16-byte aligned), each read as one 64-bit access.
__device__ __forceinline__ void ld_words2(const uint64_t *p, uint64_t &a, uint64_t &b) {
  asm volatile("ld.relaxed.gpu.global.v2.b64 {%0, %1}, [%2];" : "=l"(a), "=l"(b) : "l"(p) : "memory");
}
__device__ __forceinline__ uint64_t ld_word(const uint64_t *p) {
  uint64_t a;
  asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(a) : "l"(p) : "memory");
  return a;
}

// Another block (or kernel) gave up a bounded wait: the words or arrivals
// this block waits for may never come, so stop waiting.
__device__ __forceinline__ bool gave_up() {
  return (*static_cast<volatile unsigned *>(&g_dev_error) & kDevErrTimeout) != 0u;
}

__device__ __forceinline__ uint2 lds_u64(uint32_t addr) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
  return v;
}

// One row's code-weighted sum over this lane's first U units (unit u at
// lbase + uoff[u]): the masked dp4a loop.  The bytes of (word & (3 << 2i)) are
// codes c = q + 1 times 4^i, dp4a'd against the activation codes into
// accumulator i; the 4^i factor is removed exactly at the end.  A unit the
// lane does not have is read at an existing unit with zero activation codes,
// so the loop has no per-unit branch.
template <int U>
__device__ __forceinline__ int row_sum(uint32_t lbase, const uint32_t (&uoff)[kUPT], const uint32_t (&xa)[kUPT][8]) {
  int a0 = 0, a1 = 0, a2 = 0, a3 = 0;
#pragma unroll
  for (int u = 0; u < U; ++u) {
    const uint2 wv = lds_u64(lbase + uoff[u]);
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

struct RowCtx {
  float cm;          // fl32(gamma / s)
  int xl;            // this lane's sum of activation codes over its units
  uint32_t laddr;    // this lane's first unit, bytes from the row start
  int rb;            // packed row bytes
  float *y;          // y + first row of the stage
  uint64_t *mb;      // output words + first row of the stage, or null
  uint32_t tag;
};

__device__ __forceinline__ void put_out(const RowCtx &x, int r, int t) {
  const float v = __fmul_rn(static_cast<float>(t), x.cm);
  x.y[r] = v;
  if (x.mb != nullptr) st_word(x.mb + r, v, x.tag);
}

// Whole rows (one warp per row): rows r0 = slot, slot + step, ... of a stage,
// two in flight per iteration (their loads and dp4a chains interleave).
template <int U>
__device__ __forceinline__ void stage_rows_whole(uint32_t sbase, int nr, int slot, int step, int lane,
                                                 const uint32_t (&uoff)[kUPT], const uint32_t (&xa)[kUPT][8],
                                                 const RowCtx &x) {
  for (int r = slot; r < nr; r += 2 * step) {
    const int r2 = r + step < nr ? r + step : r;
    int t0 = row_sum<U>(sbase + static_cast<uint32_t>(r * x.rb) + x.laddr, uoff, xa) - x.xl;
    int t1 = row_sum<U>(sbase + static_cast<uint32_t>(r2 * x.rb) + x.laddr, uoff, xa) - x.xl;
    t0 = __reduce_add_sync(0xffffffffu, t0);
    t1 = __reduce_add_sync(0xffffffffu, t1);
    if (lane == 0) put_out(x, r, t0);
    if (lane == 1 && r2 != r) put_out(x, r2, t1);
  }
}

// Rows split over G warps: warp chunk `cid` of rows slot, slot + step, ...;
// the chunks' sums meet in shared memory and the last arriver writes.
template <int U>
__device__ __forceinline__ void stage_rows_split(uint32_t sbase, int nr, int slot, int step, int lane, int G,
                                                 int32_t *part, uint32_t *cnt, const uint32_t (&uoff)[kUPT],
                                                 const uint32_t (&xa)[kUPT][8], const RowCtx &x) {
  for (int r = slot; r < nr; r += step) {
    int t = row_sum<U>(sbase + static_cast<uint32_t>(r * x.rb) + x.laddr, uoff, xa) - x.xl;
    t = __reduce_add_sync(0xffffffffu, t);
    if (lane == 0) {
      atomicAdd(&part[r], t);
      __threadfence_block();
      if (atomicAdd(&cnt[r], 1u) == static_cast<uint32_t>(G - 1)) {
        __threadfence_block();
        const int tot = atomicExch(&part[r], 0);
        cnt[r] = 0u;
        put_out(x, r, tot);
      }
    }
  }
}

// Rows of call c owned by this block: [r0, r0 + rows).
__device__ __forceinline__ void block_rows(const Call &c, int &r0, int &rows) {
  r0 = static_cast<int>(blockIdx.x) * c.rpc;
  rows = c.N - r0 < c.rpc ? c.N - r0 : c.rpc;
  if (rows < 0) rows = 0;
}
__device__ __forceinline__ int row_bytes_of(int K) { return ((K + 63) / 64) * 16; }

// Eight activations of vector v (elements 8v .. 8v+7) into f; false when
// they come from output words and one of them does not carry `want` yet.
__device__ __forceinline__ bool load_vec8(const Call &c, int v, uint32_t want, float (&f)[8]) {
  if (c.mb_in != nullptr) {
    uint64_t w[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) ld_words2(c.mb_in + 8 * v + 2 * i, w[2 * i], w[2 * i + 1]);
    bool ok = true;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      ok &= static_cast<uint32_t>(w[i] >> 32) == want;
      f[i] = __uint_as_float(static_cast<uint32_t>(w[i]));
    }
    return ok;
  }
  if (c.flags & kFlagBf16) {
    const uint4 u = __ldcg(reinterpret_cast<const uint4 *>(c.x) + v);
    const uint32_t ww[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      f[2 * e] = __uint_as_float(ww[e] << 16);
      f[2 * e + 1] = __uint_as_float(ww[e] & 0xFFFF0000u);
    }
  } else {
    const float4 f0 = __ldcg(reinterpret_cast<const float4 *>(c.x) + 2 * v);
    const float4 f1 = __ldcg(reinterpret_cast<const float4 *>(c.x) + 2 * v + 1);
    f[0] = f0.x; f[1] = f0.y; f[2] = f0.z; f[3] = f0.w;
    f[4] = f1.x; f[5] = f1.y; f[6] = f1.z; f[7] = f1.w;
  }
  return true;
}

// Element k of the input; false when it comes from an output word that does
// not carry `want` yet.
__device__ __forceinline__ bool load_one(const Call &c, int k, uint32_t want, float &f) {
  if (c.mb_in != nullptr) {
    const uint64_t w = ld_word(c.mb_in + k);
    f = __uint_as_float(static_cast<uint32_t>(w));
    return static_cast<uint32_t>(w >> 32) == want;
  }
  f = (c.flags & kFlagBf16) ? __bfloat162float(__ldcg(static_cast<const __nv_bfloat16 *>(c.x) + k))
                            : __ldcg(static_cast<const float *>(c.x) + k);
  return true;
}

__device__ __forceinline__ float act_of(const Call &c, float v) {
  return (c.flags & kFlagRelu2) ? relu2f(v) : v;
}

__device__ __forceinline__ void put_codes8(uint32_t xs, int v, const float (&f)[8], float s) {
  uint32_t lo = 0, hi = 0;
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    lo |= (static_cast<uint32_t>(quant_one(f[e], s)) & 0xFFu) << (8 * e);
    hi |= (static_cast<uint32_t>(quant_one(f[e + 4], s)) & 0xFFu) << (8 * e);
  }
  sts_u64(xs + 8 * v, lo, hi);
}

__global__ void __maxnreg__(120) chain_kernel(const __grid_constant__ Params p) {
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
    sm.seq_tag = p.ctl[kCtlSeq] << 9;  // tags: (launch sequence << 9) | (call + 1)
    fence_barrier_init();
  }
  {
    const uint32_t *src = reinterpret_cast<const uint32_t *>(p.c);
    uint32_t *dst = reinterpret_cast<uint32_t *>(sm.calls);
    const int words = p.n * static_cast<int>(sizeof(Call) / 4);
    for (int w = tid; w < words; w += kThreads) dst[w] = src[w];
    for (int i = tid; i < kStages * kMaxSplitRows; i += kThreads) {
      (&sm.part[0][0])[i] = 0;
      (&sm.cnt[0][0])[i] = 0u;
    }
  }
  __syncthreads();
  volatile int *abort_flag = &sm.abort_flag;
  const uint32_t seq_tag = sm.seq_tag;

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
        for (int q = 0; q < rows; q += c.stage_rows, ++i) {
          const int s = i % kStages;
          if (i >= kStages && (!mbar_wait(smem_u32(&sm.empty[s]), ((i / kStages) - 1) & 1) || *abort_flag)) {
            *abort_flag = 1;
            go = false;
            break;
          }
          const int nr = rows - q < c.stage_rows ? rows - q : c.stage_rows;
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
  } else {
    // -------------------------------------------------- consumers
    int it = 0;       // ring stage counter, in the producer's order
    int nbar = 0;     // grid barriers passed
    // Every consumer warp passes the same sequence of block barriers: a
    // decision to stop is taken only from a barrier's reduced predicate (the
    // same in every warp); a warp that stops streaming rows early still runs
    // the later calls' barriers.
    for (int ci = 0; ci < p.n; ++ci) {
      const Call &c = sm.calls[ci];
      const float gam = __ldg(c.gamma);  // static input: fetched early
      int r0, rows;
      block_rows(c, r0, rows);

      if (c.flags & kFlagBarrier) {
        // every consumer warp of this block is done with the earlier calls;
        // thread 0's release covers their stores (cumulativity), and the
        // acquire it then takes is shared with the block by the next barrier
        ++nbar;
        named_bar(1, kC);
        bool late = false;
        if (tid == 0) {
          red_release_add(p.ctl + kCtlBar, 1u);
          const unsigned target = static_cast<unsigned>(nbar) * gridDim.x;
          const long long t0 = clock64();
          while (ld_acquire(p.ctl + kCtlBar) < target) {
            if (clock64() - t0 > kWaitLimitCycles || *abort_flag || gave_up()) {
              atomicOr(&g_dev_error, kDevErrTimeout);
              late = true;
              break;
            }
          }
        }
        if (named_bar_or(1, kC, late)) {
          *abort_flag = 1;
          break;
        }
      }
      if (rows == 0) continue;

      // ---- the input: per-token absmax, s, c = gamma / s, codes in shared memory
      const int rb = row_bytes_of(c.K);
      const int units = rb / 8;
      const int kp = rb * 4;
      const uint32_t want = seq_tag | static_cast<uint32_t>(c.src + 1);
      const bool vec = (c.K % 8) == 0 &&
                       (c.mb_in != nullptr ? (reinterpret_cast<uintptr_t>(c.mb_in) & 15u) == 0u
                                           : (reinterpret_cast<uintptr_t>(c.x) & 15u) == 0u);
      const int nv = vec ? c.K / 8 : 0;
      const bool in_regs = nv <= kJM * kC;
      float xv[kJM][8];
      bool timed_out = false;
      float a = 0.0f;
      {
        // first pass: every value (polling output words until they carry the
        // producing call's tag); kept in registers when they fit
        const long long t0 = clock64();
        for (int v0 = tid; v0 < nv; v0 += kJM * kC) {
          bool ok[kJM];
#pragma unroll
          for (int j = 0; j < kJM; ++j) {
            const int v = v0 + j * kC;
            ok[j] = v < nv ? load_vec8(c, v, want, xv[j]) : true;
            if (v >= nv)
#pragma unroll
              for (int e = 0; e < 8; ++e) xv[j][e] = 0.0f;
          }
          bool all = true;
#pragma unroll
          for (int j = 0; j < kJM; ++j) all &= ok[j];
          while (!all) {
            if (clock64() - t0 > kWaitLimitCycles || gave_up()) {
              timed_out = true;
              break;
            }
            all = true;
#pragma unroll
            for (int j = 0; j < kJM; ++j)
              if (!ok[j]) {
                ok[j] = load_vec8(c, v0 + j * kC, want, xv[j]);
                all &= ok[j];
              }
          }
#pragma unroll
          for (int j = 0; j < kJM; ++j)
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              xv[j][e] = act_of(c, xv[j][e]);
              a = fmaxf(a, fabsf(xv[j][e]));
            }
          if (timed_out) break;
        }
        for (int k = 8 * nv + tid; k < c.K && !timed_out; k += kC) {
          float f;
          while (!load_one(c, k, want, f)) {
            if (clock64() - t0 > kWaitLimitCycles || gave_up()) {
              timed_out = true;
              break;
            }
          }
          a = fmaxf(a, fabsf(act_of(c, f)));
        }
      }
      if (timed_out) atomicOr(&g_dev_error, kDevErrTimeout);
      a = warp_max_nonneg(a);
      if (lane == 0) sm.fred[warp] = a;
      if (named_bar_or(1, kC, timed_out || *abort_flag)) {
        *abort_flag = 1;
        break;
      }
      a = sm.fred[0];
#pragma unroll
      for (int w = 1; w < kCW; ++w) a = fmaxf(a, sm.fred[w]);
      const float s = act_scale(a);
      // codes (every value is present now: a second pass reads plainly)
      if (in_regs) {
#pragma unroll
        for (int j = 0; j < kJM; ++j) {
          const int v = tid + j * kC;
          if (v < nv) put_codes8(xs, v, xv[j], s);
        }
      } else {
        for (int v = tid; v < nv; v += kC) {
          float f[8];
          load_vec8(c, v, want, f);
#pragma unroll
          for (int e = 0; e < 8; ++e) f[e] = act_of(c, f[e]);
          put_codes8(xs, v, f, s);
        }
      }
      for (int k = 8 * nv + tid; k < kp; k += kC) {
        int q = 0;
        if (k < c.K) {
          float f;
          load_one(c, k, want, f);
          q = quant_one(act_of(c, f), s);
        }
        sts_u8(xs + k, static_cast<uint32_t>(q) & 0xFFu);
      }
      named_bar(1, kC);

      // ---- this warp's chunk of K: activation codes in registers, and the
      // lane's share of X = sum of codes (sum c*x - X = sum q*x, lane by lane)
      const int G = 1 << c.split_log2;
      const int cid = warp & (G - 1);
      const int slot = warp >> c.split_log2;
      const int step = kCW >> c.split_log2;
      const int ubase = cid * c.chunk;
      const int uend = ubase + c.chunk < units ? ubase + c.chunk : units;
      uint32_t xa[kUPT][8];
      uint32_t uoff[kUPT];
      int xl = 0;
      const bool lane_in = ubase + lane < uend;  // otherwise every unit is read at the chunk's first
#pragma unroll
      for (int u = 0; u < kUPT; ++u) {
        const int unit = ubase + lane + 32 * u;
        uint4 lo4 = make_uint4(0u, 0u, 0u, 0u), hi4 = lo4;
        uoff[u] = 0u;
        if (unit < uend) {
          lo4 = lds_u128(xs + 32 * unit);
          hi4 = lds_u128(xs + 32 * unit + 16);
          uoff[u] = 256u * u;
        }
        xa[u][0] = lo4.x; xa[u][1] = lo4.y; xa[u][2] = lo4.z; xa[u][3] = lo4.w;
        xa[u][4] = hi4.x; xa[u][5] = hi4.y; xa[u][6] = hi4.z; xa[u][7] = hi4.w;
#pragma unroll
        for (int e = 0; e < 8; ++e) xl = dp4a_us(0x01010101u, xa[u][e], xl);
      }
      const int upt = (c.chunk + 31) / 32;  // unit slots this call needs
      RowCtx x;
      x.cm = __fdiv_rn(gam, s);
      x.xl = xl;
      x.laddr = 8u * static_cast<uint32_t>(lane_in ? ubase + lane : ubase);
      x.rb = rb;
      x.tag = seq_tag | static_cast<uint32_t>(ci + 1);
      // (xs is rewritten by the next call only after its first block barrier)

      // ---- rows, stage by stage
      for (int q = 0; q < rows; q += c.stage_rows, ++it) {
        const int st = it % kStages;
        if (*abort_flag || !mbar_wait(smem_u32(&sm.full[st]), (it / kStages) & 1)) {
          *abort_flag = 1;
          break;
        }
        const int nr = rows - q < c.stage_rows ? rows - q : c.stage_rows;
        const uint32_t sbase = ring + st * kStageBytes;
        x.y = c.y + r0 + q;
        x.mb = c.mb_out != nullptr ? c.mb_out + r0 + q : nullptr;
        if (G == 1) {
          switch (upt) {
#define BL_W(U) case U: stage_rows_whole<U>(sbase, nr, slot, step, lane, uoff, xa, x); break;
            BL_W(1) BL_W(2) BL_W(3) BL_W(4) BL_W(5) BL_W(6) BL_W(7)
            default: stage_rows_whole<8>(sbase, nr, slot, step, lane, uoff, xa, x); break;
#undef BL_W
          }
        } else {
          switch (upt) {
#define BL_S(U) case U: stage_rows_split<U>(sbase, nr, slot, step, lane, G, sm.part[st], sm.cnt[st], uoff, xa, x); break;
            BL_S(1) BL_S(2) BL_S(3) BL_S(4) BL_S(5) BL_S(6) BL_S(7)
            default: stage_rows_split<8>(sbase, nr, slot, step, lane, G, sm.part[st], sm.cnt[st], uoff, xa, x); break;
#undef BL_S
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&sm.empty[st]));
      }
    }
  }

  // ---- the block is done with the launch; the last block to finish resets
  // the counters and advances the sequence number for the next launch (each
  // warp reconverges first: the producer's lane 0 may still be streaming)
  __syncwarp();
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    if (atomicAdd(p.ctl + kCtlDone, 1u) == gridDim.x - 1) {
      p.ctl[kCtlBar] = 0u;
      p.ctl[kCtlDone] = 0u;
      p.ctl[kCtlSeq] = p.ctl[kCtlSeq] + 1u;
      __threadfence();
    }
  }
}

}  // namespace chain
}  // namespace bl
