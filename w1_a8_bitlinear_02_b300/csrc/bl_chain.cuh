// Decode chain: a sequence of BitLinear forwards of 1 to 16 tokens in one
// persistent launch.  A call may read an earlier call's output as its input.
//
// A decode step runs the projections of every layer one after another
// ("BitNet b1.58 2B4T" architecture: QKV, O, FFN up, FFN down per layer;
// "20亿参数仅0.4GB…「原生1.58bit」大模型", blog.csdn.net/soaring_casia,
// section 2).  As separate launches each call pays a kernel boundary although
// its packed weights -- static inputs -- are a fraction of a microsecond of
// HBM time.  Here one block per SM stays resident for the whole chain:
//   * its four producer threads stream the block's rows of every call, call
//     after call, into one ring of shared-memory stages by TMA (stage i is
//     producer i mod 4's): the weights of later calls arrive while earlier
//     calls compute, limited only by the ring's size ("pack-store-load-
//     unpack-compute", 微软AI大模型炸场：0.4GB, blog.csdn.net/2401_84494441,
//     section 3, GPU bullet, carried across calls);
//   * the 16 consumer warps, in two teams of 8, run the calls in order over
//     the block's rows.
//
// Rows, one lane each.  A call's rows form groups of 32 consecutive rows,
// dealt out to the blocks round-robin, each call's deal continuing where the
// previous call's ended, so the lanes are full and the blocks' loads even out
// over the chain.  A stage is a group and a slab of its packed bytes: P
// 16-byte pieces (64 weights each) of every row, P odd and at most 65 (1040
// bytes, 4160 weights; the row's slabs as even as that allows), loaded as ONE
// TMA box of 2P 8-byte elements x 32 rows.  Rows land P * 16
// bytes apart, an odd number of 16-byte units, so the 8 lanes of a
// quarter-warp reading piece p of their own rows touch 8 different bank
// groups with no swizzle; and one copy per stage keeps the producer's issue
// cost (a TMA instruction waits behind the consumers' shared-memory traffic)
// to two instructions per stage with the record's.
// Row groups alternate between the two teams; the 8 warps of a team split
// each slab's pieces by class (piece p mod 8, rotated from call to call);
// every lane of a warp needs the same 64 activation codes, which are
// broadcast from shared memory.  A lane adds its row's pieces with the
// masked dp4a (the bytes of (word & (3 << 2i)) are the codes c = q + 1 times
// 4^i; the 4^i factor is removed exactly at the end; sum c*x - X = sum q*x,
// X = the warp's sum of activation codes) across all slabs of the group; the
// team's partial sums then meet in shared memory once per group and one warp
// writes y = fl32(acc * c), c = fl32(gamma / s).  No per-row reduction, no
// copy of the activation codes per warp, and K of any length splits the same
// way.  Calls of 2-4 tokens share the code planes across the tokens' dp4a;
// calls of 5-16 tokens run their pieces on the int8 mma.sync form.
//
// The activation codes (per-token absmax, "20亿参数仅0.4GB" page, section 2,
// item 2) of a call come one of two ways:
//   * an input no earlier call writes is quantised before the chain starts
//     (chain_setup_kernel, one block per such call and token) into a record in the
//     workspace -- codes, c and the 16 warps' code sums -- and each weight
//     stage carries the record's codes for its slab (and, for a group's first
//     slab, the header), so these calls stream with no per-call set-up;
//   * an input an earlier call writes is quantised by every block when the
//     call comes up, into a shared-memory area of its own.
//
// Dependencies between calls come in two forms, both found by the host from
// the calls' buffers:
//   * output words: when a call's x lies inside an earlier call's y, that
//     earlier call also writes each output as one 8-byte word {value, tag}
//     into the workspace, and the reader polls those words directly: the tag
//     says the value is there, so no barrier, fence or separate flag is needed
//     (an aligned 64-bit store is seen whole or not at all).  The tag holds the
//     producing call and a per-launch sequence number kept in the workspace,
//     so words left by an earlier launch never match;
//   * grid barrier: any other overlap (an input read from memory that an
//     earlier call wrote, an output that overwrites an earlier input or
//     output) makes every block finish all earlier calls first (one release-add
//     per block on a counter, acquire-spin until all have arrived).
// All blocks must be resident at once (they may wait for each other): the
// launch is cooperative, one block per SM.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cstdint>
#include <type_traits>

#include "bl_pack_quant.cuh"
#include "bl_ptx.cuh"

namespace bl {
namespace chain {

constexpr int kMaxCalls = 240;            // one tensor map each in the kernel parameters
constexpr int kCW = 16;                   // consumer warps
constexpr int kTeams = 2;                 // one-token row groups alternate between two teams
constexpr int kTW = kCW / kTeams;         // warps of a team
constexpr int kProd = 4;                  // producer warps (one thread each): stage i is producer i mod kProd's
constexpr int kThreads = (kCW + kProd) * 32;
constexpr int kC = kCW * 32;              // consumer threads
constexpr int kMaxK = 32768;
constexpr int kMaxN = 1 << 30;            // row indices stay far inside int
constexpr int kGroupRows = 32;            // rows per group at most: one per lane
constexpr int kPiece = 16;                // packed bytes of a piece (64 weights)
constexpr int kJM = 2;                    // x vectors of 8 per consumer thread kept in registers (K <= 8192)
// Pieces per slab: odd (conflict-free rows, see above), at most 65 for one
// token, 31 for 2-8 and 23 for 9-16 (their stage also holds every token's
// codes); a row
// of np pieces takes the fewest slabs the cap allows, split evenly.
__host__ __device__ constexpr int piece_cap(int M) { return M > 8 ? 23 : (M > 1 ? 31 : 65); }
__host__ __device__ constexpr int slab_pieces(int rb, int M = 1) {
  return ((rb / kPiece + (rb / kPiece + piece_cap(M) - 1) / piece_cap(M) - 1) /
          ((rb / kPiece + piece_cap(M) - 1) / piece_cap(M))) | 1;
}
__host__ __device__ constexpr int slabs_of(int rb, int M = 1) {
  return (rb / kPiece + slab_pieces(rb, M) - 1) / slab_pieces(rb, M);
}
// A record in the workspace: a 128-byte header -- c = gamma / s (fp32) at
// byte 0, the code sums of the 16 piece classes (slab piece p mod 16; int32)
// at byte 64 -- then the codes, zero from K to the end of the last slab.  The
// in-block codes area has the same header (c only) and the codes zero to the
// end of the row's last piece.
constexpr int kHeader = 128;
constexpr int kInBlockBytes = kHeader + kMaxK;
// A ring stage: the slab's weights (32 rows of P pieces), then at codes_ofs
// the record header and the slab's activation codes (one bulk copy for a
// group's first slab, whose header travels with it).
__host__ __device__ constexpr int codes_ofs(int M) { return kGroupRows * kPiece * piece_cap(M); }
constexpr int kStageBytes = 37 * 1024;
// Ring stages: five in the one-token streaming form (no many-token call, no
// input quantised in the block), whose fixed region is small and which needs
// no in-block codes area; four in the other forms.
constexpr int kStagesMax = 5;
__host__ __device__ constexpr int stages_of(bool many, bool dep) { return (!many && !dep) ? 5 : 4; }
// Token rows of the group-sum buffers: every token of a many-token call, else
// the two teams' one-token sums (see Item).
__host__ __device__ constexpr int sum_rows(bool many) { return many ? 16 : 2; }
// Barriers, partial sums and the call table.
__host__ __device__ constexpr int smem_fixed(bool many) { return (many ? 45 : 31) * 1024; }
__host__ __device__ constexpr int smem_bytes(bool many, bool dep) {
  return 1024 + smem_fixed(many) + stages_of(many, dep) * kStageBytes + (dep ? kInBlockBytes : 0);
}

// Control words at the start of the workspace (bytes 0..255), then the
// call table, the records, the output words.
constexpr int kCtlBar = 0;    // grid-barrier arrivals of this launch
constexpr int kCtlDone = 1;   // blocks finished with this launch
constexpr int kCtlSeq = 32;   // launches completed on this workspace (tags)
constexpr int kTableOffset = 256;

// Call flags.
constexpr int kFlagBf16 = 1;      // x is bf16 (else fp32)
constexpr int kFlagRelu2 = 2;     // quantise relu2(x)
constexpr int kFlagBarrier = 4;   // every block finishes all earlier calls first

// Calls of more than one token (up to kMaxTok) use slabs of at most 31 (23)
// pieces, so a stage holds the weights (at most 15.5 KB) and every token's
// codes for them (M x 31 x 64 bytes); their record header holds c[m] (fp32)
// at 4m and the 16 warps' code sums of token m at 64 + 64m.
constexpr int kMaxTok = 16;
constexpr int kMmaTok = 5;  // calls of kMmaTok..kMaxTok tokens run their pieces on the tensor cores
constexpr int kDp4aTok = kMmaTok - 1;  // 2..kDp4aTok tokens on dp4a
__host__ __device__ constexpr int header_bytes(int M) { return M > 1 ? ((64 + 64 * M + 127) / 128) * 128 : kHeader; }
// a record: the header, then slab by slab each token's codes (64 per piece)
__host__ __device__ constexpr int record_bytes(int rb, int M = 1) {
  return header_bytes(M) + slabs_of(rb, M) * M * 64 * slab_pieces(rb, M);
}
static_assert(codes_ofs(1) + kHeader + 64 * piece_cap(1) <= kStageBytes, "a stage of a one-token call");
static_assert(codes_ofs(8) + header_bytes(8) + 8 * 64 * piece_cap(8) <= kStageBytes, "a stage of 8 tokens");
static_assert(codes_ofs(kMaxTok) + header_bytes(kMaxTok) + kMaxTok * 64 * piece_cap(kMaxTok) <= kStageBytes,
              "a stage of a many-token call");
static_assert(kStageBytes % 1024 == 0 && codes_ofs(1) % 128 == 0 && codes_ofs(8) % 128 == 0 &&
                  codes_ofs(kMaxTok) % 128 == 0,
              "stage and codes alignment");

struct Call {
  const float *gamma;
  const void *x;          // [K] f32 or bf16 (read when neither rec nor mb_in is set)
  float *y;               // [N]
  const uint8_t *rec;     // the call's quantised input (record), or null
  uint64_t *mb_out;       // this call's output words [N] {value bits, tag}, or null
  const uint64_t *mb_in;  // the words holding x [K] (inside an earlier call's mb_out), or null
  int N, K;
  int rb;                 // packed row bytes
  int g0;                 // the block that takes group 0 (group j goes to block (g0 + j) mod grid)
  int ng;                 // 32-row groups: ceil(N / 32)
  int flags;
  int src;                // the call that wrote mb_in
  int M;                  // tokens (x [M, K], y [M, N]); more than one only with a record
  int P;                  // pieces per slab (slab_pieces(rb, M); the box is 4P words wide)
  int ns;                 // slabs per row (slabs_of(rb, M))
};
static_assert(sizeof(Call) % 4 == 0, "call table copied in words");

// The packed weights of call i are read through maps[i]: [N, rb / 8] 8-byte
// elements, box 2P elements x 32 rows, no swizzle, zeros outside.  Tensor maps in
// the kernel parameters need no fetch from global memory (a map read from
// global memory stalled the issuing thread by about an L2 round trip per
// call).
struct Params {
  int n;                  // calls
  unsigned *ctl;          // workspace control words
  const Call *table;      // the call table (in the workspace)
  CUtensorMap maps[kMaxCalls];
};

// Row sums of one-token groups meet in one of kGB buffers, each with an
// mbarrier the group's warps arrive on once their shares are added; only the
// warp that writes the group's rows waits.  No warp can be kStages + 1 groups
// ahead of another (each group takes at least one stage), so kGB > kStagesMax + 1
// keeps a buffer from being reused before its group is written.
constexpr int kGB = 8;
static_assert(kGB > kStagesMax + 1, "group buffers");
static_assert(kGB % kTeams == 0 && kCW % kTeams == 0, "teams");
static_assert(kThreads <= 20 * 32, "the kernel's register budget assumes at most 20 warps");

// This block's share of a call, built once per launch: the first of its
// row groups (j0), how many it takes (cnt: j0, j0 + grid, ... below the
// call's group count), N, and packed: pieces per slab (bits 0-7), slabs per
// row (8-15), pieces per row (16-25), tokens - 1 (26-29), kCbFast (30: one
// token, input quantised ahead, no barrier) and kCbRec (31: a record).
struct __align__(16) CallBlk {
  int j0, cnt, N;
  uint32_t pk;
};
constexpr uint32_t kCbFast = 1u << 30;
constexpr uint32_t kCbRec = 1u << 31;
static_assert(piece_cap(1) < 256 && piece_cap(2) < 256 && piece_cap(kMaxTok) < 256 &&
                  slabs_of(kPiece * (kMaxK / 64), 1) < 256 && slabs_of(kPiece * (kMaxK / 64), 2) < 256 &&
                  slabs_of(kPiece * (kMaxK / 64), kMaxTok) < 256 && kMaxK / 64 < 1024 && kMaxTok <= 16,
              "CallBlk::pk's fields hold the largest call");

// When every call of the chain takes the fast form (one token, input
// quantised ahead, no barrier), the producers hand the block's row groups to
// the two teams through one queue per team (group o of the block goes to
// team o mod 2 as its entry o / 2; seq = entry + 1 once written, released
// after the other fields), so the consumers read one entry per group and
// never walk the call table.  A queue slot is rewritten only kTQ entries
// later, after its group was summed: no stage is issued before the stage
// kStages earlier was released, so the producers run at most kStages stages
// ahead of the oldest stage a team still holds.
struct __align__(16) Item {
  float *y;
  uint64_t *mbo;  // output words, or null
  int it;         // the group's first ring stage
  int r0;         // its first row
  int N;
  uint32_t pk;    // CallBlk::pk of the call
  int ci;         // the call
  int seq;
  int pad[2];
};
constexpr int kTQ = 16;
constexpr int kTB = 8;  // group-sum buffers per team (a team's warps are at most kStages of its groups apart)

template <bool MANY>
struct SmemT {
  uint64_t full[kStagesMax];
  uint64_t empty[kStagesMax];
  uint64_t gbar[kGB];
  float fred[kCW];
  int xcls[2][kCW];  // code sums of in-block inputs by piece class (p mod 16), by call parity
  int32_t gsum[kGB][sum_rows(MANY)][kGroupRows];  // by group buffer, token, row
  float gcm[kGB][sum_rows(MANY)];                 // the tokens' output scales c, by group buffer
  uint32_t seq_tag;
  int abort_flag;
  int stage_tag[kStagesMax];  // the stage each ring slot was last armed for (written by the producer that armed it)
  CallBlk cb[kMaxCalls];  // this block's share of each call
  Item tq[kTeams][kTQ];   // the teams' group queues (every call in the fast form)
  uint64_t tbar[kTeams][kTB];  // their group-sum barriers (the sums in gsum, flat)
  int tq_end[kTeams];     // the number of groups of each team
  int ib[kMaxCalls];      // each call's first ring stage in this block
  int og[kMaxCalls];      // and the block's ordinal of its first group
  uint32_t scan_w[kThreads / 32][2];
  Call calls[kMaxCalls];  // the call table, copied in once
};
static_assert(sizeof(Item) == 48, "queue entry");
static_assert(kTeams * kTB <= kGB * sum_rows(false), "team sums inside gsum");
static_assert(kMaxTok <= sum_rows(true), "every token's sums");
static_assert(sizeof(CallBlk) == 16, "one 16-byte load a call");
static_assert(sizeof(SmemT<false>) <= smem_fixed(false) && sizeof(SmemT<true>) <= smem_fixed(true),
              "fixed shared-memory region");
static_assert(smem_bytes(false, false) <= 227 * 1024 && smem_bytes(false, true) <= 227 * 1024 &&
                  smem_bytes(true, false) <= 227 * 1024 && smem_bytes(true, true) <= 227 * 1024,
              "shared memory of one block");

// ------------------------------------------------------------ set-up kernels
// The set-up launch before each chain: the call table into the workspace
// (its parameters hold the table by value, so a captured graph keeps it; each
// block copies a slice), then the inputs no earlier call writes quantised
// into their records: token m of x [M, K] (f32 or bf16, relu2 first if
// flagged) -> its part of the record (c[m] = gamma / s_m, the code sums of
// the 16 piece classes, codes zero-padded to the last slab).  Grid (calls,
// most tokens); block (i, m) takes token m of call i if it has a record.
struct TableCopy {
  int n;
  Call *dst;
  Call calls[kMaxCalls];
};
constexpr int kQThreads = 512;
__global__ void __launch_bounds__(kQThreads) chain_setup_kernel(const __grid_constant__ TableCopy q) {
  __shared__ __align__(16) uint8_t codes[kMaxK + 64 * piece_cap(1)];
  __shared__ float red[kQThreads / 32];
  __shared__ int xsum[kCW];
  pdl_launch_dependents();  // the chain may set up its barriers meanwhile
  {
    const uint32_t *src = reinterpret_cast<const uint32_t *>(q.calls);
    uint32_t *dst = reinterpret_cast<uint32_t *>(q.dst);
    const int words = q.n * static_cast<int>(sizeof(Call) / 4);
    const int nb = static_cast<int>(gridDim.x * gridDim.y);
    const int b = static_cast<int>(blockIdx.y * gridDim.x + blockIdx.x);
    for (int i = b * kQThreads + static_cast<int>(threadIdx.x); i < words; i += nb * kQThreads) dst[i] = src[i];
  }
  struct {
    const void *x;
    const float *gamma;
    uint8_t *rec;
    int K, rb, flags, M, P;
  } jb;
  {
    const Call &c = q.calls[blockIdx.x];
    jb = {c.x, c.gamma, const_cast<uint8_t *>(c.rec), c.K, c.rb, c.flags, c.M, c.P};
  }
  const int m = blockIdx.y;
  if (jb.rec == nullptr || m >= jb.M) return;
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const bool bf = (jb.flags & kFlagBf16) != 0, r2 = (jb.flags & kFlagRelu2) != 0;
  const int K = jb.K, M = jb.M, P = jb.P, SB4 = 64 * P, nsl = slabs_of(jb.rb, M), kend = nsl * SB4;
  const void *xr = bf ? static_cast<const void *>(static_cast<const __nv_bfloat16 *>(jb.x) + static_cast<int64_t>(m) * K)
                      : static_cast<const void *>(static_cast<const float *>(jb.x) + static_cast<int64_t>(m) * K);
  auto ld = [&](int k) -> float {
    const float v = bf ? __bfloat162float(static_cast<const __nv_bfloat16 *>(xr)[k]) : static_cast<const float *>(xr)[k];
    return r2 ? relu2f(v) : v;
  };
  const bool vec = (K % 8) == 0 && al16(xr);
  const int nv = vec ? K / 8 : 0;
  if (vec && nv <= 2 * kQThreads) {
    // one read of x, kept in registers; each thread writes its vectors' codes
    // straight into the record, and the 8 lanes holding one 64-code piece
    // add its sum into the piece's class
    const float gam = t == 0 ? __ldg(jb.gamma) : 0.0f;
    float f[2][8];
    float a = 0.0f;
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const int v = t + r * kQThreads;
      if (v < nv) {
        if (bf)
          load8(static_cast<const __nv_bfloat16 *>(xr) + 8 * v, f[r]);
        else
          load8(static_cast<const float *>(xr) + 8 * v, f[r]);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          if (r2) f[r][e] = relu2f(f[r][e]);
          a = fmaxf(a, fabsf(f[r][e]));
        }
      }
    }
    a = warp_max_nonneg(a);
    if (lane == 0) red[warp] = a;
    if (t < kCW) xsum[t] = 0;
    __syncthreads();
    a = red[0];
#pragma unroll
    for (int w = 1; w < kQThreads / 32; ++w) a = fmaxf(a, red[w]);
    const float s = act_scale(a);
    const int H = header_bytes(M);
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const int v = t + r * kQThreads;  // lanes 8i..8i+7 hold one piece (kQThreads is a multiple of 8)
      int sum = 0, cls = 0;
      if (v < nv) {
        uint32_t lo = 0, hi = 0;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          lo |= (static_cast<uint32_t>(quant_one(f[r][e], s)) & 0xFFu) << (8 * e);
          hi |= (static_cast<uint32_t>(quant_one(f[r][e + 4], s)) & 0xFFu) << (8 * e);
        }
        const int k = 8 * v, sl = k / SB4, off = k - sl * SB4;
        *reinterpret_cast<uint2 *>(jb.rec + H + (static_cast<size_t>(sl) * M + m) * SB4 + off) = make_uint2(lo, hi);
        sum = dp4a_us(0x01010101u, hi, dp4a_us(0x01010101u, lo, 0));
        cls = (off / 64) % kCW;
      }
      sum += __shfl_xor_sync(0xffffffffu, sum, 1);
      sum += __shfl_xor_sync(0xffffffffu, sum, 2);
      sum += __shfl_xor_sync(0xffffffffu, sum, 4);
      if ((lane & 7) == 0 && v < nv) atomicAdd(&xsum[cls], sum);
    }
    // zeros from K to the end of the last slab
    for (int k = 8 * (nv + t); k < kend; k += 8 * kQThreads) {
      const int sl = k / SB4, off = k - sl * SB4;
      *reinterpret_cast<uint2 *>(jb.rec + H + (static_cast<size_t>(sl) * M + m) * SB4 + off) = make_uint2(0u, 0u);
    }
    __syncthreads();
    if (t < kCW) reinterpret_cast<int *>(jb.rec + 64 + 64 * m)[t] = xsum[t];
    if (t == 0) reinterpret_cast<float *>(jb.rec)[m] = __fdiv_rn(gam, s);
    return;
  }
  float a = 0.0f;
  for (int v = t; v < nv; v += kQThreads) {
    float f[8];
    if (bf)
      load8(static_cast<const __nv_bfloat16 *>(xr) + 8 * v, f);
    else
      load8(static_cast<const float *>(xr) + 8 * v, f);
#pragma unroll
    for (int e = 0; e < 8; ++e) a = fmaxf(a, fabsf(r2 ? relu2f(f[e]) : f[e]));
  }
  for (int k = 8 * nv + t; k < K; k += kQThreads) a = fmaxf(a, fabsf(ld(k)));
  a = warp_max_nonneg(a);
  if (lane == 0) red[warp] = a;
  if (t < kCW) xsum[t] = 0;
  __syncthreads();
  a = red[0];
#pragma unroll
  for (int w = 1; w < kQThreads / 32; ++w) a = fmaxf(a, red[w]);
  const float s = act_scale(a);
  for (int v = t; v < nv; v += kQThreads) {
    float f[8];
    if (bf)
      load8(static_cast<const __nv_bfloat16 *>(xr) + 8 * v, f);
    else
      load8(static_cast<const float *>(xr) + 8 * v, f);
    uint32_t lo = 0, hi = 0;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      lo |= (static_cast<uint32_t>(quant_one(r2 ? relu2f(f[e]) : f[e], s)) & 0xFFu) << (8 * e);
      hi |= (static_cast<uint32_t>(quant_one(r2 ? relu2f(f[e + 4]) : f[e + 4], s)) & 0xFFu) << (8 * e);
    }
    *reinterpret_cast<uint2 *>(codes + 8 * v) = make_uint2(lo, hi);
  }
  for (int k = 8 * nv + t; k < kend; k += kQThreads)
    codes[k] = k < K ? static_cast<uint8_t>(quant_one(ld(k), s) & 0xFF) : 0u;
  __syncthreads();
  // the codes out, slab by slab after the header (token m's share of each
  // slab), and each 64-code piece's sum into its warp's total (piece p of a
  // slab is read by consumer warp p mod 16)
  const int H = header_bytes(M);
  for (int i = t; i < kend / 16; i += kQThreads) {
    const int sl = (16 * i) / SB4, off = (16 * i) % SB4;
    *reinterpret_cast<uint4 *>(jb.rec + H + (static_cast<size_t>(sl) * M + m) * SB4 + off) =
        *reinterpret_cast<const uint4 *>(codes + 16 * i);
  }
  for (int pc = t; pc < kend / 64; pc += kQThreads) {
    int sm = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint4 v = *reinterpret_cast<const uint4 *>(codes + 64 * pc + 16 * i);
      sm = dp4a_us(0x01010101u, v.x, sm);
      sm = dp4a_us(0x01010101u, v.y, sm);
      sm = dp4a_us(0x01010101u, v.z, sm);
      sm = dp4a_us(0x01010101u, v.w, sm);
    }
    atomicAdd(&xsum[(pc % P) % kCW], sm);
  }
  __syncthreads();
  if (t < kCW) reinterpret_cast<int *>(jb.rec + 64 + 64 * m)[t] = xsum[t];
  if (t == 0) reinterpret_cast<float *>(jb.rec)[m] = __fdiv_rn(__ldg(jb.gamma), s);
}

// ------------------------------------------------------------ helpers
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

// Wait for ring stage `it` to land.  A parity wait on a slot is only sound
// once the slot's previous stage (it - kStages) has landed: before that, the
// phase two back has the same parity and the wait would pass at once.  A
// warp that processed stage it - kStages saw it land (bit kStages - 1 of
// `seen`, the warp's record of which of the last kStages stages it
// processed); a warp that skipped it (another team's row group) first waits
// for the slot to be armed for `it`, which happens only after the slot's
// previous stage was consumed.  Bounded; false when the block must stop.
template <int kStages>
__device__ __forceinline__ bool stage_ready(const uint64_t *full, const int *stage_tag, int it, uint32_t seen,
                                            volatile int *abort_flag) {
  const int st = it % kStages;
  if (!(seen & (1u << (kStages - 1)))) {
    const long long t0 = clock64();
    while (true) {
      int tag;
      asm volatile("ld.acquire.cta.shared.s32 %0, [%1];" : "=r"(tag) : "r"(smem_u32(&stage_tag[st])) : "memory");
      if (tag == it) break;
      if (*abort_flag || clock64() - t0 > kWaitLimitCycles || gave_up()) {
        atomicOr(&g_dev_error, kDevErrTimeout);
        return false;
      }
    }
  }
  const uint32_t bar = smem_u32(&full[st]);
  if (mbar_try_wait(bar, (it / kStages) & 1)) return true;
  return !*abort_flag && mbar_wait_slow(bar, (it / kStages) & 1);
}

// This block's first group of call c (it takes groups j, j + grid, ...;
// none when j >= c.ng).
__device__ __forceinline__ int first_group(const Call &c) {
  const int j = static_cast<int>(blockIdx.x) - c.g0;
  return j < 0 ? j + static_cast<int>(gridDim.x) : j;
}
// Pieces of slab s that lie inside the row (the last slab may be shorter).
__device__ __forceinline__ int pieces_in(int rb, int P, int s) {
  const int left = rb / kPiece - s * P;
  return left < P ? left : P;
}

// Eight activations of vector v into f; false when they come from output
// words and one of them does not carry `want` yet.
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

// Codes of vector v into the codes area; returns their sum.
__device__ __forceinline__ int put_codes8(uint32_t xs, int v, const float (&f)[8], float s) {
  uint32_t lo = 0, hi = 0;
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    lo |= (static_cast<uint32_t>(quant_one(f[e], s)) & 0xFFu) << (8 * e);
    hi |= (static_cast<uint32_t>(quant_one(f[e + 4], s)) & 0xFFu) << (8 * e);
  }
  sts_u64(xs + 8 * v, lo, hi);
  return dp4a_us(0x01010101u, hi, dp4a_us(0x01010101u, lo, 0));
}

// Vectors of 8 the call's input is read in (0: element by element).
__device__ __forceinline__ int vec_count(const Call &c) {
  const bool vec = (c.K % 8) == 0 && (c.mb_in != nullptr ? (reinterpret_cast<uintptr_t>(c.mb_in) & 15u) == 0u
                                                          : (reinterpret_cast<uintptr_t>(c.x) & 15u) == 0u);
  return vec ? c.K / 8 : 0;
}

// One 16-byte piece of a lane's row (64 weights) against the 64 activation
// codes at `act` (broadcast): accumulator i gets the bit-plane-i codes x 4^i.
__device__ __forceinline__ void piece(uint32_t waddr, uint32_t act, int (&a)[4]) {
  const uint4 w = lds_u128(waddr);
  const uint4 x0 = lds_u128(act), x1 = lds_u128(act + 16), x2 = lds_u128(act + 32), x3 = lds_u128(act + 48);
  const uint32_t wd[4] = {w.x, w.y, w.z, w.w};
  const uint32_t xv[16] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w,
                           x2.x, x2.y, x2.z, x2.w, x3.x, x3.y, x3.z, x3.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    a[0] = dp4a_us(wd[j] & 0x03030303u, xv[4 * j + 0], a[0]);
    a[1] = dp4a_us(wd[j] & 0x0C0C0C0Cu, xv[4 * j + 1], a[1]);
    a[2] = dp4a_us(wd[j] & 0x30303030u, xv[4 * j + 2], a[2]);
    a[3] = dp4a_us(wd[j] & 0xC0C0C0C0u, xv[4 * j + 3], a[3]);
  }
}

// The pieces of one stage of a one-token group taken by this warp: class
// pcls, pcls + STEP, ..., two at a time in separate accumulators so their
// loads and dp4a chains overlap.
template <int STEP>
__device__ __forceinline__ void stage_one(uint32_t sbase, uint32_t abase, int pcls, int npc, int (&acc)[4],
                                          int (&acc2)[4]) {
  int pc = pcls;
  for (; pc + STEP < npc; pc += 2 * STEP) {
    piece(sbase + static_cast<uint32_t>(pc * kPiece), abase + 64u * pc, acc);
    piece(sbase + static_cast<uint32_t>((pc + STEP) * kPiece), abase + 64u * (pc + STEP), acc2);
  }
  if (pc < npc) piece(sbase + static_cast<uint32_t>(pc * kPiece), abase + 64u * pc, acc);
}

// Quantise the input of call c in every block that has rows of it (it
// depends on earlier calls) into the in-block codes area `slot`: values
// polled from output words or read after the grid barrier, per-token absmax
// over the block, codes zero-padded to the end of the row's last piece and
// c = gamma / s into the area's header; xw = the code sum of piece class cls
// (slab pieces p with p mod 16 == cls), added up per class while the codes
// are written (nq: the block's count of such calls, picking the class-sum
// buffer).  Returns false (in every thread) when the block must stop.
template <class Smem>
__device__ __forceinline__ bool quantise_in_block(const Call &c, uint32_t slot, uint32_t want, int tid, int cls,
                                                  int nq, Smem &sm, volatile int *abort_flag, int &xw) {
  const int warp = tid >> 5, lane = tid & 31;
  const uint32_t xs = slot + kHeader;
  const int nv = vec_count(c);
  const bool in_regs = nv <= kJM * kC;
  const float gam = __ldg(c.gamma);  // off the critical path: needed after the last value arrives
  int *const xcls = sm.xcls[nq & 1];  // last used two such calls ago
  const int P = c.P;
  float xv[kJM][8];
  bool timed_out = false;
  float a = 0.0f;
  const long long t0 = clock64();
  // first pass: every value (polling output words until they carry the
  // producing call's tag); kept in registers when they fit
  for (int v0 = tid; v0 < nv; v0 += kJM * kC) {
    bool ok[kJM];
#pragma unroll
    for (int j = 0; j < kJM; ++j) {
      const int v = v0 + j * kC;
      if (v < nv) {
        ok[j] = load_vec8(c, v, want, xv[j]);
      } else {
        ok[j] = true;
#pragma unroll
        for (int e = 0; e < 8; ++e) xv[j][e] = 0.0f;
      }
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
  if (timed_out) atomicOr(&g_dev_error, kDevErrTimeout);
  a = warp_max_nonneg(a);
  if (lane == 0) sm.fred[warp] = a;
  if (tid < kCW) xcls[tid] = 0;
  if (named_bar_or(1, kC, timed_out || *abort_flag)) return false;
  a = sm.fred[0];
#pragma unroll
  for (int w = 1; w < kCW; ++w) a = fmaxf(a, sm.fred[w]);
  const float s = act_scale(a);
  // codes (every value is present now: a second pass reads plainly), then
  // zeros from K to the end of the last slab
  // (vector v lies in global piece v / 8, slab piece (v / 8) mod P)
  if (in_regs) {
#pragma unroll
    for (int j = 0; j < kJM; ++j) {
      const int v = tid + j * kC;
      if (v < nv) atomicAdd(&xcls[((v >> 3) % P) & (kCW - 1)], put_codes8(xs, v, xv[j], s));
    }
  } else {
    for (int v = tid; v < nv; v += kC) {
      float f[8];
      load_vec8(c, v, want, f);
#pragma unroll
      for (int e = 0; e < 8; ++e) f[e] = act_of(c, f[e]);
      atomicAdd(&xcls[((v >> 3) % P) & (kCW - 1)], put_codes8(xs, v, f, s));
    }
  }
  const int kz = (c.K + 15) & ~15;
  for (int k = 8 * nv + tid; k < kz; k += kC) {
    int q = 0;
    if (k < c.K) {
      float f;
      load_one(c, k, want, f);
      q = quant_one(act_of(c, f), s);
      atomicAdd(&xcls[((k >> 6) % P) & (kCW - 1)], q);
    }
    sts_u8(xs + k, static_cast<uint32_t>(q) & 0xFFu);
  }
  for (int k = kz + 16 * tid; k < 4 * c.rb; k += 16 * kC) sts_u128(xs + k, 0u, 0u, 0u, 0u);
  if (tid == 0) asm volatile("st.shared.f32 [%0], %1;" ::"r"(slot), "f"(__fdiv_rn(gam, s)) : "memory");
  named_bar(1, kC);
  xw = xcls[cls];
  return true;
}

// One 16-byte piece against MT tokens' activation codes (token m's 64 codes
// at act + m * tstride, broadcast): the codes are shifted down once per word
// and shared by the tokens; acc[m] += sum c * x.
template <int MT>
__device__ __forceinline__ void piece_multi(uint32_t waddr, uint32_t act, uint32_t tstride, int (&acc)[kDp4aTok]) {
  const uint4 w = lds_u128(waddr);
  const uint32_t wd[4] = {w.x, w.y, w.z, w.w};
  uint32_t cw[16];
#pragma unroll
  for (int j = 0; j < 4; ++j)
#pragma unroll
    for (int i = 0; i < 4; ++i) cw[4 * j + i] = (wd[j] >> (2 * i)) & 0x03030303u;
#pragma unroll
  for (int m = 0; m < MT; ++m) {
    const uint32_t at = act + m * tstride;
    const uint4 x0 = lds_u128(at), x1 = lds_u128(at + 16), x2 = lds_u128(at + 32), x3 = lds_u128(at + 48);
    const uint32_t xv[16] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w,
                             x2.x, x2.y, x2.z, x2.w, x3.x, x3.y, x3.z, x3.w};
#pragma unroll
    for (int t = 0; t < 16; ++t) acc[m] = dp4a_us(cw[t], xv[t], acc[m]);
  }
}

// The pieces of one stage of a many-token call (this warp's: class cls,
// cls + kTW, ...).
template <int MT>
__device__ __forceinline__ void stage_multi(uint32_t sbase, uint32_t abase, uint32_t tstride, int npc, int cls,
                                            int (&acc)[kDp4aTok]) {
  for (int pc = cls; pc < npc; pc += kTW)
    piece_multi<MT>(sbase + static_cast<uint32_t>(pc * kPiece), abase + 64u * pc, tstride, acc);
}

// The pieces of one stage of a call of 5-8 tokens on the tensor cores
// (legacy mma.sync, m16n8k32, u8 codes x s8 activation codes -> exact s32):
// this warp's 16-row tile (trow = the tile's first row in the stage) and
// piece class pcls (p mod 4).  Lane (g, t) = (lane / 4, lane % 4) holds word t
// of rows g and g + 8 of each piece; plane i of a word (its bytes masked by
// 3 << 2i, shifted down) is four codes c = q + 1 for k = 16t + 4i .. 16t + 4i + 3,
// so planes 0-1 feed one MMA's A (fragment k 4t.. and 16 + 4t..) and planes
// 2-3 the next; B is the same k range of token g's codes (one 16-byte load),
// the 8 MMA columns being the tokens (columns past M are discarded).
// d[4u + 0..1]: row g, tokens 8u + 2t, 8u + 2t + 1; d[4u + 2..3]: row g + 8
// (u: the token tile, NT tiles of 8 tokens, sharing the weight fragments;
// tile u's codes are act + 8u * tstride).
template <int NT>
__device__ __forceinline__ void stage_mma(uint32_t trow, uint32_t act, uint32_t tstride, int npc, int pcls, int P,
                                          int lane, int (&d)[8]) {
  const int g = lane >> 2, t = lane & 3;
  const uint32_t ra = trow + static_cast<uint32_t>(g * kPiece * P + 4 * t);
  const uint32_t rbo = ra + static_cast<uint32_t>(8 * kPiece * P);
  const uint32_t xa = act + static_cast<uint32_t>(16 * t);
  for (int pc = pcls; pc < npc; pc += 4) {
    uint32_t wa, wb;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(wa) : "r"(ra + static_cast<uint32_t>(pc * kPiece)));
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(wb) : "r"(rbo + static_cast<uint32_t>(pc * kPiece)));
    uint4 x[NT];
#pragma unroll
    for (int u = 0; u < NT; ++u) x[u] = lds_u128(xa + 8u * u * tstride + 64u * pc);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint32_t a0 = (wa >> (4 * h)) & 0x03030303u, a2 = (wa >> (4 * h + 2)) & 0x03030303u;
      const uint32_t a1 = (wb >> (4 * h)) & 0x03030303u, a3 = (wb >> (4 * h + 2)) & 0x03030303u;
#pragma unroll
      for (int u = 0; u < NT; ++u) {
        const uint32_t b0 = h ? x[u].z : x[u].x, b1 = h ? x[u].w : x[u].y;
        asm volatile(
            "mma.sync.aligned.m16n8k32.row.col.s32.u8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
            : "+r"(d[4 * u + 0]), "+r"(d[4 * u + 1]), "+r"(d[4 * u + 2]), "+r"(d[4 * u + 3])
            : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
      }
    }
  }
}

// MANY: the chain has calls of more than one token (a separate instantiation,
// so single-token chains keep their register budget).
// The register budget is set as for 20 warps (at most 96 registers a thread):
// with 18 warps, two of the four schedulers hold 5 warps, and each
// scheduler's share of the register file must fit 5 x 32 x the count.
// DEP: the chain has calls whose input is quantised in the block (an
// earlier call writes it); only those take the all-warps form of a group,
// so chains without them keep the streaming form's register allocation.
template <bool MANY, bool DEP>
__global__ void __launch_bounds__(20 * 32, 1) chain_kernel(const __grid_constant__ Params p) {
  constexpr int kStages = stages_of(MANY, DEP);
  using Smem = SmemT<MANY>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;  // stages start 1 KB aligned (TMA needs 128 bytes)
  Smem &sm = *reinterpret_cast<Smem *>(smem_raw + (base - raw));
  const uint32_t ring = base + smem_fixed(MANY);
  const uint32_t inb = ring + kStages * kStageBytes;  // codes quantised in this block
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&sm.full[s]), 1);
      mbar_init(smem_u32(&sm.empty[s]), kCW);
    }
    for (int b = 0; b < kGB; ++b) mbar_init(smem_u32(&sm.gbar[b]), kCW);
    for (int t = 0; t < kTeams; ++t) {
      for (int b = 0; b < kTB; ++b) mbar_init(smem_u32(&sm.tbar[t][b]), kTW);
      for (int k = 0; k < kTQ; ++k) sm.tq[t][k].seq = 0;
      sm.tq_end[t] = -1;
    }
    sm.abort_flag = 0;
    for (int s = 0; s < kStages; ++s) sm.stage_tag[s] = s;
    fence_barrier_init();
  }
  // the set-up launch writes the call table and the records: wait for it (a
  // no-op when the launch does not overlap it)
  pdl_wait_primary();
  if (tid == 0) sm.seq_tag = p.ctl[kCtlSeq] << 9;  // tags: (launch sequence << 9) | (call + 1)
  {
    const uint32_t *src = reinterpret_cast<const uint32_t *>(p.table);
    uint32_t *dst = reinterpret_cast<uint32_t *>(sm.calls);
    const int words = p.n * static_cast<int>(sizeof(Call) / 4);
    for (int w = tid; w < words; w += kThreads) dst[w] = src[w];
    for (int i = tid; i < static_cast<int>(sizeof(sm.gsum) / 4); i += kThreads) (&sm.gsum[0][0][0])[i] = 0;
  }
  __syncthreads();
  // this block's share of each call (one thread a call), then the calls'
  // first stages and group ordinals in the block (prefix sums over the calls)
  static_assert(kMaxCalls <= kThreads, "one thread a call");
  bool mine_fast = true;
  uint32_t vs = 0, vg = 0;  // the call's stages and groups in this block
  if (tid < p.n) {
    const int i = tid;
    const Call &c = sm.calls[i];
    const int G = static_cast<int>(gridDim.x);
    int j0 = static_cast<int>(blockIdx.x) - c.g0;
    if (j0 < 0) j0 += G;
    CallBlk e;
    e.j0 = j0;
    e.cnt = j0 < c.ng ? (c.ng - j0 + G - 1) / G : 0;
    e.N = c.N;
    const bool fast = c.M == 1 && c.rec != nullptr && (c.flags & kFlagBarrier) == 0;
    e.pk = static_cast<uint32_t>(c.P) | (static_cast<uint32_t>(c.ns) << 8) |
           (static_cast<uint32_t>(c.rb / kPiece) << 16) | (static_cast<uint32_t>(c.M - 1) << 26) |
           (fast ? kCbFast : 0u) | (c.rec != nullptr ? kCbRec : 0u);
    sm.cb[i] = e;
    mine_fast = fast;
    vs = static_cast<uint32_t>(e.cnt) * static_cast<uint32_t>(c.ns);
    vg = static_cast<uint32_t>(e.cnt);
  }
  {
    uint32_t is = vs, ig = vg;  // inclusive prefix sums within the warp
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const uint32_t a = __shfl_up_sync(0xffffffffu, is, d), b = __shfl_up_sync(0xffffffffu, ig, d);
      if (lane >= d) {
        is += a;
        ig += b;
      }
    }
    if (lane == 31) {
      sm.scan_w[warp][0] = is;
      sm.scan_w[warp][1] = ig;
    }
    __syncthreads();
    if (tid < p.n) {
      for (int w = 0; w < warp; ++w) {
        is += sm.scan_w[w][0];
        ig += sm.scan_w[w][1];
      }
      sm.ib[tid] = static_cast<int>(is - vs);
      sm.og[tid] = static_cast<int>(ig - vg);
      if (tid == p.n - 1) {
        sm.tq_end[0] = static_cast<int>((ig + 1) / 2);
        sm.tq_end[1] = static_cast<int>(ig / 2);
      }
    }
  }
  const bool qmode = __syncthreads_and(mine_fast) != 0 && !MANY && !DEP;
  volatile int *abort_flag = &sm.abort_flag;
  const uint32_t seq_tag = sm.seq_tag;

  if (warp >= kCW) {
    // ------------------------------------------------ producers: records and weight stages.
    // Stage i of the block is issued by producer i mod kProd into ring slot
    // i mod kStages; each producer takes up only the calls that hold one of
    // its stages (from the stage prefix sums), so the per-call and per-stage
    // issue work is spread over kProd threads on different schedulers.  A
    // slot's stages may belong to different producers, so a producer first
    // waits until the slot was armed for its previous stage (the slot's tag)
    // and only then waits on that stage's empty phase: never a parity wait
    // two phases behind.
    static_assert((kProd & (kProd - 1)) == 0, "stage owner by mask");
    const int q = warp - kCW;
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      const uint64_t pol_rec = policy_evict_last();  // records are read by every block
      int issued = 0;
      bool go = true;
      // the call's fields in registers, read one call ahead (shared-memory
      // loads wait behind the consumers' traffic; the asm statements below
      // clobber memory, which would make every later use a reload)
      struct Fields {
        uint4 e;  // CallBlk
        int ib, og;
        const uint8_t *rec;
        float *y;
        uint64_t *mbo;
      };
      auto fields = [&](int ci) {
        Fields f;
        f.e = lds_u128(smem_u32(&sm.cb[ci]));
        f.ib = sm.ib[ci];
        f.og = sm.og[ci];
        f.rec = sm.calls[ci].rec;
        f.y = qmode ? sm.calls[ci].y : nullptr;
        f.mbo = qmode ? sm.calls[ci].mb_out : nullptr;
        return f;
      };
      Fields nxt = fields(0);
      for (int ci = 0; ci < p.n && go; ++ci) {
        const Fields cur = nxt;
        if (ci + 1 < p.n) nxt = fields(ci + 1);
        const int cnt = static_cast<int>(cur.e.y);
        const uint32_t pk = cur.e.w;
        const int nslab = static_cast<int>((pk >> 8) & 0xFFu), len = cnt * nslab;
        const int d = (q - cur.ib) & (kProd - 1);  // this producer's first stage of the call, from its first
        if (d >= len) continue;
        const int M = static_cast<int>((pk >> 26) & 0xFu) + 1, P = static_cast<int>(pk & 0xFFu);
        const int G = static_cast<int>(gridDim.x);
        const uint8_t *rec = cur.rec;
        const int H = header_bytes(M);
        const uint32_t cbytes = static_cast<uint32_t>(M * 64 * P);  // every token's codes of one slab
        const uint32_t cofs = static_cast<uint32_t>(codes_ofs(M));
        const CUtensorMap *map = &p.maps[ci];
        // this block's groups j0, j0 + G, ... (the last group may run past N,
        // where the box reads zeros; so does the last slab past the row)
        const uint32_t box = static_cast<uint32_t>(kGroupRows * kPiece * P);
        int g = d / nslab, s = d - g * nslab;  // the stage's group (of the block's) and slab
        for (int i = cur.ib + d; i < cur.ib + len; i += kProd) {
          const int j = static_cast<int>(cur.e.x) + g * G;
          const int st = i % kStages;
          bool armed = true;
          if (i >= kStages) {
            const long long t0 = clock64();
            while (true) {
              int tag;
              asm volatile("ld.acquire.cta.shared.s32 %0, [%1];" : "=r"(tag) : "r"(smem_u32(&sm.stage_tag[st])) : "memory");
              if (tag == i - kStages) break;
              if (*abort_flag || clock64() - t0 > kWaitLimitCycles || gave_up()) {
                atomicOr(&g_dev_error, kDevErrTimeout);
                armed = false;
                break;
              }
            }
          }
          if (i >= kStages && (!armed || !mbar_wait(smem_u32(&sm.empty[st]), ((i / kStages) - 1) & 1) || *abort_flag)) {
            *abort_flag = 1;
            go = false;
            break;
          }
          const uint32_t fb = smem_u32(&sm.full[st]);
          const uint32_t sb = ring + st * kStageBytes;
          uint32_t tx = box;
          if (rec != nullptr) tx += cbytes + (s == 0 ? H : 0);
          mbar_arrive_expect_tx(fb, tx);
          tma_load_2d(sb, map, s * P * (kPiece / 8), j * kGroupRows, fb, pol);
          if (rec != nullptr) {
            if (s == 0)
              bulk_g2s(sb + cofs, rec, H + cbytes, fb, pol_rec);
            else
              bulk_g2s(sb + cofs + H, rec + H + s * cbytes, cbytes, fb, pol_rec);
          }
          if (i >= kStages)
            asm volatile("st.release.cta.shared.s32 [%0], %1;" ::"r"(smem_u32(&sm.stage_tag[st])), "r"(i) : "memory");
          if (qmode && s == 0) {
            // the group's queue entry (its slot's previous entry was
            // consumed: see Item)
            const int o = cur.og + g, k = o >> 1;
            Item &e = sm.tq[o & 1][k % kTQ];
            e.y = cur.y;
            e.mbo = cur.mbo;
            e.it = i;
            e.r0 = j * kGroupRows;
            e.N = static_cast<int>(cur.e.z);
            e.pk = pk;
            e.ci = ci;
            asm volatile("st.release.cta.shared.s32 [%0], %1;" ::"r"(smem_u32(&e.seq)), "r"(k + 1) : "memory");
          }
          issued = i + 1;
          s += kProd;
          while (s >= nslab) {
            s -= nslab;
            ++g;
          }
        }
      }
      // no copy into this block's shared memory may be in flight at exit:
      // done once stage j landed, or once its slot was armed again (which
      // needs stage j consumed; never a parity wait two phases behind)
      for (int j = issued - kStages < 0 ? 0 : issued - kStages; j < issued; ++j)
        if (j % kProd == q) {
          const uint32_t bar = smem_u32(&sm.full[j % kStages]);
          const long long t0 = clock64();
          while (!mbar_try_wait(bar, (j / kStages) & 1)) {
            if (*static_cast<volatile int *>(&sm.stage_tag[j % kStages]) != j) break;
            if (clock64() - t0 > kWaitLimitCycles) {
              atomicOr(&g_dev_error, kDevErrTimeout);
              break;
            }
          }
        }
    }
    __syncwarp();
  } else {
    // -------------------------------------------------- consumers
    // Every consumer warp passes the same sequence of block barriers: a
    // decision to stop is taken only from a barrier's reduced predicate (the
    // same in every warp); a warp that stops streaming early still runs the
    // later calls' barriers.
    int it = 0;       // ring stage counter, in the producer's order
    int nbar = 0;     // grid barriers passed
    int ng1 = 0;      // row groups done (team, group buffer, writer and phase)
    int nq = 0;       // calls whose input this block quantised
    uint32_t seen = (1u << kStages) - 1u;  // bit b: this warp processed stage it - 1 - b (stages before 0 count as seen)
    if (qmode) {
      // ---- every call in the fast form: this team's groups from its queue
      const int team = warp / kTW, tw = warp % kTW;
      int last = -1;  // the last stage this warp processed
      int *const tsum = &sm.gsum[0][0][0];
      for (int k = 0;; ++k) {
        const Item &E = sm.tq[team][k % kTQ];
        bool end = false;
        {
          const long long t0 = clock64();
          while (true) {
            int sq, en;
            asm volatile("ld.acquire.cta.shared.s32 %0, [%1];" : "=r"(sq) : "r"(smem_u32(&E.seq)) : "memory");
            if (sq == k + 1) break;
            asm volatile("ld.acquire.cta.shared.s32 %0, [%1];" : "=r"(en) : "r"(smem_u32(&sm.tq_end[team])) : "memory");
            if (en == k) {
              end = true;
              break;
            }
            if (*abort_flag || clock64() - t0 > kWaitLimitCycles || gave_up()) {
              atomicOr(&g_dev_error, kDevErrTimeout);
              *abort_flag = 1;
              end = true;
              break;
            }
          }
        }
        if (end) break;
        const int it0 = E.it, r0 = E.r0, N = E.N, ci = E.ci;
        const uint32_t pk = E.pk;
        float *const yout = E.y;
        uint64_t *const mbo = E.mbo;
        const int P = static_cast<int>(pk & 0xFFu), nslab = static_cast<int>((pk >> 8) & 0xFFu);
        const int np = static_cast<int>((pk >> 16) & 0x3FFu);
        const int cls = (tw + ci) & (kTW - 1);
        const uint32_t lrow = static_cast<uint32_t>(lane * kPiece * P);
        const int gap = it0 - last - 1;  // the other team's stages since this warp's last one
        seen = gap >= 32 ? 0u : seen << gap;
        int acc[4] = {0, 0, 0, 0}, acc2[4] = {0, 0, 0, 0};
        float cm = 0.0f;
        int xw = 0;
        for (int s = 0; s < nslab; ++s) {
          const int it = it0 + s, st = it % kStages;
          if (!stage_ready<kStages>(sm.full, sm.stage_tag, it, seen, abort_flag)) {
            *abort_flag = 1;
            break;
          }
          seen = (seen << 1) | 1u;
          const int left = np - s * P;
          const int npc = left < P ? left : P;
          const uint32_t sb = ring + st * kStageBytes;
          if (s == 0) {
            uint32_t x0, x1;
            asm volatile("ld.shared.f32 %0, [%1];" : "=f"(cm) : "r"(sb + codes_ofs(1)) : "memory");
            asm volatile("ld.shared.u32 %0, [%1];" : "=r"(x0) : "r"(sb + codes_ofs(1) + 64u + 4u * cls) : "memory");
            asm volatile("ld.shared.u32 %0, [%1];" : "=r"(x1) : "r"(sb + codes_ofs(1) + 64u + 4u * (cls + kTW))
                         : "memory");
            xw = static_cast<int>(x0 + x1);
          }
          stage_one<kTW>(sb + lrow, sb + codes_ofs(1) + kHeader, cls, npc, acc, acc2);
          __syncwarp();
          if (lane == 0) mbar_arrive_n(smem_u32(&sm.empty[st]), static_cast<uint32_t>(kTeams));
        }
        last = it0 + nslab - 1;
        // the team's sums meet in buffer k mod kTB; warp k mod kTW writes the rows
        const int b = k & (kTB - 1);
        int *const sum = tsum + (team * kTB + b) * kGroupRows;
        atomicAdd(sum + lane, (acc[0] + acc2[0]) + ((acc[1] + acc2[1]) >> 2) + ((acc[2] + acc2[2]) >> 4) +
                                  ((acc[3] + acc2[3]) >> 6) - xw);
        __syncwarp();
        if (lane == 0) mbar_arrive_n(smem_u32(&sm.tbar[team][b]), 1u);
        if (tw == (k % kTW) && !*abort_flag) {
          if (mbar_wait(smem_u32(&sm.tbar[team][b]), (k / kTB) & 1)) {
            const int t = sum[lane];
            sum[lane] = 0;
            const int r = r0 + lane;
            if (r < N) {
              const float v = __fmul_rn(static_cast<float>(t), cm);
              yout[r] = v;
              if (mbo != nullptr) st_word(mbo + r, v, seq_tag | static_cast<uint32_t>(ci + 1));
            }
          } else {
            *abort_flag = 1;
          }
        }
      }
    }
    for (int ci = 0; ci < (qmode ? 0 : p.n); ++ci) {
      {
        // ---- one token, input quantised ahead, no barrier: the block's
        // share of the call from one 16-byte entry; this team's groups are
        // every other one of the block's (group ng1 + g goes to team
        // (ng1 + g) mod 2), the other team's stages are stepped over
        const uint4 e = lds_u128(smem_u32(&sm.cb[ci]));
        if (e.w & kCbFast) {
          const int cnt = static_cast<int>(e.y);
          if (cnt == 0) continue;
          const int G = static_cast<int>(gridDim.x), N = static_cast<int>(e.z);
          const int P = static_cast<int>(e.w & 0xFFu), nslab = static_cast<int>((e.w >> 8) & 0xFFu);
          const int np = static_cast<int>((e.w >> 16) & 0x3FFu);
          float *const yout = sm.calls[ci].y;
          uint64_t *const mbo = sm.calls[ci].mb_out;
          const int team = warp / kTW, tw = warp % kTW;
          const int cls = (tw + ci) & (kTW - 1);
          const uint32_t lrow = static_cast<uint32_t>(lane * kPiece * P);
          const uint32_t tag = seq_tag | static_cast<uint32_t>(ci + 1);
          const uint32_t skip_seen = nslab >= 32 ? 0u : ~0u;
          int g = (ng1 ^ team) & 1;
          if (g != 0) {  // the block's first group of the call is the other team's
            it += nslab;
            seen = (seen << (nslab & 31)) & skip_seen;
          }
          for (; g < cnt; g += 2) {
            const int o = ng1 + g;  // the group's ordinal in the block
            int acc[4] = {0, 0, 0, 0}, acc2[4] = {0, 0, 0, 0};
            float cm = 0.0f;
            int xw = 0;
            for (int s = 0; s < nslab; ++s, ++it) {
              const int st = it % kStages;
              if (!stage_ready<kStages>(sm.full, sm.stage_tag, it, seen, abort_flag)) {
                *abort_flag = 1;
                break;
              }
              seen = (seen << 1) | 1u;
              const int left = np - s * P;
              const int npc = left < P ? left : P;
              const uint32_t sb = ring + st * kStageBytes;
              if (s == 0) {
                // c and X of class cls (the header holds the sums of the 16
                // classes p mod 16; classes cls and cls + kTW make p mod kTW)
                uint32_t x0, x1;
                asm volatile("ld.shared.f32 %0, [%1];" : "=f"(cm) : "r"(sb + codes_ofs(1)) : "memory");
                asm volatile("ld.shared.u32 %0, [%1];" : "=r"(x0) : "r"(sb + codes_ofs(1) + 64u + 4u * cls) : "memory");
                asm volatile("ld.shared.u32 %0, [%1];" : "=r"(x1) : "r"(sb + codes_ofs(1) + 64u + 4u * (cls + kTW))
                             : "memory");
                xw = static_cast<int>(x0 + x1);
              }
              stage_one<kTW>(sb + lrow, sb + codes_ofs(1) + kHeader, cls, npc, acc, acc2);
              // the stage's empty barrier counts kCW arrivals: a team's warps
              // arrive twice each
              __syncwarp();
              if (lane == 0) mbar_arrive_n(smem_u32(&sm.empty[st]), static_cast<uint32_t>(kTeams));
            }
            const int gb = o & (kGB - 1);
            atomicAdd(&sm.gsum[gb][0][lane], (acc[0] + acc2[0]) + ((acc[1] + acc2[1]) >> 2) +
                                              ((acc[2] + acc2[2]) >> 4) + ((acc[3] + acc2[3]) >> 6) - xw);
            __syncwarp();  // orders the lanes' adds before lane 0's release
            if (lane == 0) mbar_arrive_n(smem_u32(&sm.gbar[gb]), static_cast<uint32_t>(kTeams));
            if (tw == ((o / kTeams) % kTW) && !*abort_flag) {
              if (mbar_wait(smem_u32(&sm.gbar[gb]), (o / kGB) & 1)) {
                const int t = sm.gsum[gb][0][lane];
                sm.gsum[gb][0][lane] = 0;
                const int r = (static_cast<int>(e.x) + g * G) * kGroupRows + lane;
                if (r < N) {
                  const float v = __fmul_rn(static_cast<float>(t), cm);
                  yout[r] = v;
                  if (mbo != nullptr) st_word(mbo + r, v, tag);
                }
              } else {
                *abort_flag = 1;
              }
            }
            if (g + 1 < cnt) {  // the other team's next group
              it += nslab;
              seen = (seen << (nslab & 31)) & skip_seen;
            }
          }
          ng1 += cnt;
          continue;
        }
      }
      const Call &c = sm.calls[ci];
      const int j0 = first_group(c), G = static_cast<int>(gridDim.x);

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
      if (j0 >= c.ng) continue;  // no group of this call here (nor its input quantisation)
      // the call's fields in registers (asm statements below clobber memory)
      const bool has_rec = c.rec != nullptr;
      const int rb = c.rb, M = c.M, N = c.N, P = c.P, ngr = c.ng;
      float *const yout = c.y;
      uint64_t *const mbo = c.mb_out;
      const uint32_t lrow = static_cast<uint32_t>(lane * kPiece * P);  // this lane's row in a stage
      // Row groups alternate between the two teams of kTW warps (group ng1
      // goes to team ng1 mod 2), so each warp takes more pieces of a stage
      // for the same per-stage work; within its team a warp takes the slab
      // pieces of class cls (p mod kTW == cls), rotated from call to call so
      // the classes with one piece more fall to different warps.  A group's
      // sums meet in a group buffer (gsum, gbar): no block barrier.
      const int team = warp / kTW, tw = warp % kTW;
      const int cls = (tw + ci) & (kTW - 1);

      if (MANY && M > 1) {
        // ---- many tokens (their codes come with the record in every stage)
        const int H = header_bytes(M), nslab = c.ns;
        const uint32_t cofs = static_cast<uint32_t>(codes_ofs(M));
        const uint32_t tstride = static_cast<uint32_t>(64 * P);
        for (int j = j0; j < ngr; j += G) {
          if ((ng1 & 1) != team) {
            it += nslab;
            seen = nslab >= 32 ? 0u : seen << nslab;
            ++ng1;
            continue;
          }
          const int r0 = j * kGroupRows;
          const int gb = ng1 & (kGB - 1);
          if (M >= kMmaTok) {
            // ---- 5-16 tokens: tensor cores, warp tw takes tile tw & 1 and
            // piece class ((tw >> 1) + call) mod 4; tokens in tiles of 8
            const int tile = tw & 1, pcls4 = ((tw >> 1) + ci) & 3;
            const int gg = lane >> 2, tt = lane & 3;
            int d[8] = {0, 0, 0, 0, 0, 0, 0, 0};
            int xs[4] = {0, 0, 0, 0};  // code sums of tokens 8u + 2tt + q over this warp's pieces (u, q)
            for (int s = 0; s < nslab; ++s, ++it) {
              const int st = it % kStages;
              if (*abort_flag || !stage_ready<kStages>(sm.full, sm.stage_tag, it, seen, abort_flag)) {
                *abort_flag = 1;
                break;
              }
              seen = (seen << 1) | 1u;
              const int npc = pieces_in(rb, P, s);
              const uint32_t sb = ring + st * kStageBytes;
              if (s == 0) {
                if (tw == 0 && lane < M)
                  asm volatile("ld.shared.f32 %0, [%1];" : "=f"(sm.gcm[gb][lane]) : "r"(sb + cofs + 4u * lane)
                               : "memory");
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                  const int m = 8 * (e >> 1) + 2 * tt + (e & 1);
                  int x = 0;
                  if (m < M) {
#pragma unroll
                    for (int c4 = 0; c4 < 4; ++c4) {
                      uint32_t v;
                      asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v)
                                   : "r"(sb + cofs + 64u + 64u * m + 4u * (pcls4 + 4 * c4)) : "memory");
                      x += static_cast<int>(v);
                    }
                  }
                  xs[e] = x;
                }
              }
              const uint32_t trow = sb + static_cast<uint32_t>(tile * 16 * kPiece * P);
              const uint32_t act = sb + cofs + static_cast<uint32_t>(H) + static_cast<uint32_t>(gg) * tstride;
              if (M > 8)
                stage_mma<2>(trow, act, tstride, npc, pcls4, P, lane, d);
              else
                stage_mma<1>(trow, act, tstride, npc, pcls4, P, lane, d);
              __syncwarp();
              if (lane == 0) mbar_arrive_n(smem_u32(&sm.empty[st]), kTeams);
            }
            const int row = tile * 16 + gg;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int m = 8 * (e >> 1) + 2 * tt + (e & 1);
              if (m < M) {
                atomicAdd(&sm.gsum[gb][m][row], d[4 * (e >> 1) + (e & 1)] - xs[e]);
                atomicAdd(&sm.gsum[gb][m][row + 8], d[4 * (e >> 1) + 2 + (e & 1)] - xs[e]);
              }
            }
          } else {
            // ---- 2-4 tokens: dp4a, the shifted code planes shared by the tokens
            int acc[kDp4aTok] = {0, 0, 0, 0};
            int xwv[kDp4aTok] = {0, 0, 0, 0};
            for (int s = 0; s < nslab; ++s, ++it) {
              const int st = it % kStages;
              if (*abort_flag || !stage_ready<kStages>(sm.full, sm.stage_tag, it, seen, abort_flag)) {
                *abort_flag = 1;
                break;
              }
              seen = (seen << 1) | 1u;
              const int npc = pieces_in(rb, P, s);
              const uint32_t sb = ring + st * kStageBytes;
              if (s == 0) {
                if (tw == 0 && lane < M)
                  asm volatile("ld.shared.f32 %0, [%1];" : "=f"(sm.gcm[gb][lane]) : "r"(sb + cofs + 4u * lane)
                               : "memory");
#pragma unroll
                for (int m = 0; m < kDp4aTok; ++m)
                  if (m < M) {
                    uint32_t x0, x1;
                    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(x0) : "r"(sb + cofs + 64u + 64u * m + 4u * cls)
                                 : "memory");
                    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(x1)
                                 : "r"(sb + cofs + 64u + 64u * m + 4u * (cls + kTW))
                                 : "memory");
                    xwv[m] = static_cast<int>(x0 + x1);
                  }
              }
              const uint32_t sbase = sb + lrow, abase = sb + cofs + static_cast<uint32_t>(H);
              switch (M) {
                case 2: stage_multi<2>(sbase, abase, tstride, npc, cls, acc); break;
                case 3: stage_multi<3>(sbase, abase, tstride, npc, cls, acc); break;
                default: stage_multi<4>(sbase, abase, tstride, npc, cls, acc); break;
              }
              __syncwarp();
              if (lane == 0) mbar_arrive_n(smem_u32(&sm.empty[st]), kTeams);
            }
#pragma unroll
            for (int m = 0; m < kDp4aTok; ++m)
              if (m < M) atomicAdd(&sm.gsum[gb][m][lane], acc[m] - xwv[m]);
          }
          // the team's sums meet in the group's buffer; its writing warp
          // waits for them, writes the rows and clears the buffer (the
          // output scales c came with the group's first stage into gcm)
          __syncwarp();
          if (lane == 0) mbar_arrive_n(smem_u32(&sm.gbar[gb]), kTeams);
          if (tw == ((ng1 / kTeams) % kTW) && !*abort_flag) {
            if (!mbar_wait(smem_u32(&sm.gbar[gb]), (ng1 / kGB) & 1)) {
              *abort_flag = 1;
              ++ng1;
              continue;
            }
            for (int m = 0; m < M; ++m) {
              const int t = sm.gsum[gb][m][lane];
              sm.gsum[gb][m][lane] = 0;
              if (r0 + lane < N)
                yout[static_cast<int64_t>(m) * N + r0 + lane] = __fmul_rn(static_cast<float>(t), sm.gcm[gb][m]);
            }
          }
          ++ng1;
        }
        continue;
      }

      // ---- the activation codes, c and the warp's code sum: from the
      // record (in each group's first stage) or quantised here.  A call whose
      // input is quantised here waits for an earlier call, so its latency
      // counts: all 16 warps take each of its groups (pieces of class p mod 16).
      const bool all = DEP && !has_rec;
      const int pcls = all ? ((warp + ci) & (kCW - 1)) : cls;
      float cm = 0.0f;
      int xw = 0;
      if (!has_rec) {
        // the area is rewritten only after the block barrier inside, which
        // every warp reaches once it is done with the earlier calls
        if (!quantise_in_block(c, inb, seq_tag | static_cast<uint32_t>(c.src + 1), tid, pcls, nq, sm, abort_flag,
                               xw)) {
          *abort_flag = 1;
          break;
        }
        ++nq;
        asm volatile("ld.shared.f32 %0, [%1];" : "=f"(cm) : "r"(inb) : "memory");
      }
      const int nslab = c.ns;
      const uint32_t tag = seq_tag | static_cast<uint32_t>(ci + 1);

      // ---- row groups: one lane per row, the slabs' pieces split over the
      // warps of the group's team (the other team moves on to its next group),
      // or over all warps (ALL); one instantiation each, so the streaming form
      // keeps its register allocation
      auto groups = [&](auto all_c) {
      constexpr bool ALL = decltype(all_c)::value;
      for (int j = j0; j < ngr; j += G) {
        if (!ALL && (ng1 & 1) != team) {
          it += nslab;
          seen = nslab >= 32 ? 0u : seen << nslab;
          ++ng1;
          continue;
        }
        int acc[4] = {0, 0, 0, 0}, acc2[4] = {0, 0, 0, 0};
        for (int s = 0; s < nslab; ++s, ++it) {
          const int st = it % kStages;
          if (!stage_ready<kStages>(sm.full, sm.stage_tag, it, seen, abort_flag)) {
            *abort_flag = 1;
            break;
          }
          seen = (seen << 1) | 1u;
          const int npc = pieces_in(rb, P, s);
          const uint32_t sb = ring + st * kStageBytes;
          const uint32_t sbase = sb + lrow;
          const uint32_t abase = !ALL ? sb + codes_ofs(1) + kHeader : inb + kHeader + static_cast<uint32_t>(s * 64 * P);
          if (!ALL && s == 0) {
            // c and X of class cls (the header holds the sums of the 16
            // classes p mod 16; classes cls and cls + kTW make p mod kTW)
            uint32_t x0, x1;
            asm volatile("ld.shared.f32 %0, [%1];" : "=f"(cm) : "r"(sb + codes_ofs(1)) : "memory");
            asm volatile("ld.shared.u32 %0, [%1];" : "=r"(x0) : "r"(sb + codes_ofs(1) + 64u + 4u * cls) : "memory");
            asm volatile("ld.shared.u32 %0, [%1];" : "=r"(x1) : "r"(sb + codes_ofs(1) + 64u + 4u * (cls + kTW))
                         : "memory");
            xw = static_cast<int>(x0 + x1);
          }
          stage_one<ALL ? kCW : kTW>(sbase, abase, pcls, npc, acc, acc2);
          // the stage's empty barrier counts kCW arrivals: a team's warps
          // arrive twice each
          __syncwarp();
          if (lane == 0) mbar_arrive_n(smem_u32(&sm.empty[st]), ALL ? 1u : static_cast<uint32_t>(kTeams));
        }
        // the warps' sums meet in the group's buffer (no block barrier: a
        // warp done with its share goes on to the next group); the writing
        // warp waits for every thread's share, writes the rows and clears
        // the buffer
        const int gb = ng1 & (kGB - 1);
        atomicAdd(&sm.gsum[gb][0][lane], (acc[0] + acc2[0]) + ((acc[1] + acc2[1]) >> 2) +
                                          ((acc[2] + acc2[2]) >> 4) + ((acc[3] + acc2[3]) >> 6) - xw);
        __syncwarp();  // orders the lanes' adds before lane 0's release
        if (lane == 0) mbar_arrive_n(smem_u32(&sm.gbar[gb]), ALL ? 1u : static_cast<uint32_t>(kTeams));
        // (once the block is stopping, nothing more is waited for or written;
        // every warp still walks the same calls, so later block barriers match)
        if ((ALL ? warp == (ng1 % kCW) : tw == ((ng1 / kTeams) % kTW)) && !*abort_flag) {
          if (!mbar_wait(smem_u32(&sm.gbar[gb]), (ng1 / kGB) & 1)) {
            *abort_flag = 1;
            ++ng1;
            continue;
          }
          const int t = sm.gsum[gb][0][lane];
          sm.gsum[gb][0][lane] = 0;
          const int r = j * kGroupRows + lane;
          if (r < N) {
            const float v = __fmul_rn(static_cast<float>(t), cm);
            yout[r] = v;
            if (mbo != nullptr) st_word(mbo + r, v, tag);
          }
        }
        ++ng1;
      }
      };
      if (all)
        groups(std::true_type{});
      else
        groups(std::false_type{});
    }
    __syncwarp();
  }

  // ---- the block is done with the launch; the last block to finish resets
  // the counters and advances the sequence number for the next launch
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
