// Host-side planning for the BitLinear forward: which kernel runs for a given
// (M, N, K), its tiling, and the workspace layout.  Pure integer logic, so
// the workspace size a caller queries is the one the call uses.
#pragma once

#include <cstddef>
#include <cstdint>

namespace bl {
namespace plan {

enum Path { kGemv = 0, kTc = 1, kSkinny = 2 };

// Reference SM count used for split-K decisions (B300: 148 SMs).  A fixed
// value keeps workspace sizes independent of the device.
constexpr int kRefSms = 148;
constexpr int kGemvStageBytes = 64 * 1024;   // upper bound of one GEMV ring stage
constexpr int kGemvMaxStages = 6;
constexpr int kGemvMaxSplitRows = 32;
constexpr int kGemvSmemFixed = 8 * 1024;
constexpr int kSmemMax = 227 * 1024;
// Few-token tensor-core kernel: cluster size bound, weight ring stages, the
// barrier block, and a shared-memory floor that keeps one block per SM (each
// block takes all 512 tensor-memory columns).
constexpr int kSkMaxCs = 8;
constexpr int kSkStageBytes = 8192;  // four 64-k tiles of 128 packed rows
constexpr int kSkMaxWs = 16;
constexpr int kSkBarsBytes = 4096;
constexpr int kSkSmemFloor = 120 * 1024;
constexpr int kSkMaxM = 64;

inline int64_t row_bytes(int64_t K) { return ((K + 63) / 64) * 16; }

inline size_t align256(size_t v) { return (v + 255) & ~static_cast<size_t>(255); }

struct Plan {
  int path = kGemv;
  int64_t M = 0, N = 0, K = 0, Kp = 0, row_bytes = 0;
  // GEMV: tokens held (1, 2, 4 or 8), 8-byte units per lane, log2 warps per
  // row, units per warp chunk, consumer warps
  int mt = 1, upt = 1, split_log2 = 0, chunk = 0, cw = 8;
  // tensor-core GEMM
  int bn = 0;
  int64_t tiles_n = 0, tiles_m = 0;
  int tiles_total = 0;
  int splits = 1, kt_per_split = 0;
  // stream-K: one block per SM (kRefSms) takes an equal share of the
  // flattened (tile, k tile) units; used when whole tiles fill the last wave
  // poorly (each tile is then shared by at most two neighbouring blocks)
  int streamk = 0, sk_grid = 0, units = 0, units_per = 0;
  // few-token kernel: blocks per cluster (K split) and k tiles per block
  int sk_cs = 1, sk_kt_per = 0;
  // workspace (bytes, 256-aligned offsets)
  size_t off_xb = 0, off_sc = 0, off_acc = 0, off_cnt = 0, off_part = 0, ws_bytes = 0;
};

// Units per lane so the activation slice stays within 64 registers
// (8 registers per unit and token).
inline int upt_max(int mt) { return mt == 1 ? 8 : (mt == 2 ? 4 : (mt == 4 ? 2 : 1)); }

// Few-token kernel: shared memory of a launch (alignment slack, the B operand
// resident for the block's k tiles, a ring of ws weight stages, the split-K
// partial sums a block receives -- cs x ceil(bn / cs) token rows of 128 int32
// -- and the barrier block) and the ring depth that fits.
inline int64_t sk_red_bytes(int bn, int cs) {
  return cs > 1 ? static_cast<int64_t>(cs) * ((bn + cs - 1) / cs) * 128 * 4 : 0;
}
inline int64_t sk_smem(int bn, int64_t kt_per, int ws, int cs) {
  return 1024 + static_cast<int64_t>(bn) * 128 * kt_per + static_cast<int64_t>(ws) * kSkStageBytes +
         sk_red_bytes(bn, cs) + kSkBarsBytes;
}
// Lanes (issuer, unpack group, tensor-memory A slot) of the few-token kernel:
// the ring depth is a multiple of them, at least two stages per lane.
inline int sk_lanes(int bn) { return bn <= 32 ? 3 : 2; }
inline int sk_ring(int bn, int64_t kt_per, int cs) {
  const int64_t room = kSmemMax - sk_smem(bn, kt_per, 0, cs);
  const int ni = sk_lanes(bn);
  int64_t ws = room / kSkStageBytes;
  if (ws > kSkMaxWs) ws = kSkMaxWs;
  ws -= ws % ni;
  return ws < 2 * ni ? 0 : static_cast<int>(ws);
}
inline int sk_launch_smem(int bn, int64_t kt_per, int cs) {
  const int64_t b = sk_smem(bn, kt_per, sk_ring(bn, kt_per, cs), cs);
  return static_cast<int>(b < kSkSmemFloor ? kSkSmemFloor : b);
}

// Few-token kernel: blocks per cluster and k tiles per block for a given
// cluster size bound; false if the B operand does not fit.
inline bool sk_split(int bn, int64_t tiles_n, int num_kt, int cs_max, int *cs, int *kt_per) {
  int c0 = tiles_n >= kRefSms ? 1 : static_cast<int>(kRefSms / tiles_n);
  if (c0 > cs_max) c0 = cs_max;
  if (c0 > num_kt) c0 = num_kt;
  if (c0 < 1) c0 = 1;
  for (int c = c0; c <= cs_max && c <= num_kt; ++c) {
    const int kp = (num_kt + c - 1) / c;
    const int cc = (num_kt + kp - 1) / kp;
    if (sk_ring(bn, kp, cc) > 0) {
      *kt_per = kp;
      *cs = cc;
      return true;
    }
  }
  return false;
}

// GEMM blocks sharing one SM at token tile bn (the kernel's tensor-memory and
// shared-memory sizes are chosen for it; bitlinear.cu checks that they agree).
inline constexpr int tc_blocks_per_sm(int bn) { return bn <= 64 ? 2 : 1; }

inline Plan make(int64_t M, int64_t N, int64_t K) {
  Plan p;
  p.M = M;
  p.N = N;
  p.K = K;
  p.row_bytes = row_bytes(K);
  p.Kp = p.row_bytes * 4;
  const int64_t units = p.row_bytes / 8;
  // One or two tokens, and three or four where the codes fit: the GEMV (its
  // dp4a loop measured faster than the few-token tensor-core kernel there,
  // up to 1.8x on the 28672 x 8192 shape at three and four tokens).
  if (M <= 4) {
    p.mt = M == 1 ? 1 : (M == 2 ? 2 : 4);
    const int64_t per_warp = 32 * static_cast<int64_t>(upt_max(p.mt));
    // warps per row: the fewest (a power of two, at most 8) whose chunks fit
    int lg = 0;
    while (lg < 3 && (units + (int64_t(1) << lg) - 1) / (int64_t(1) << lg) > per_warp) ++lg;
    const int64_t chunk = (units + (int64_t(1) << lg) - 1) >> lg;
    const int64_t kp_bytes = M * p.Kp;
    if (chunk <= per_warp && kp_bytes <= 64 * 1024) {
      p.path = kGemv;
      p.split_log2 = lg;
      p.chunk = static_cast<int>(chunk);
      p.upt = static_cast<int>((chunk + 31) / 32);
      p.ws_bytes = 0;
      return p;
    }
  }
  // A few tokens: the few-token tensor-core kernel when its clusters cover
  // the weights in one wave of blocks (one per SM).  With more blocks than
  // SMs its per-block latency repeats per wave, and the GEMM below (shared
  // activation quantisation, stream-K or split-K over all SMs) measured
  // faster: 1.3-1.8x on 6912 x 2560 at 64 tokens and on the 28672 x 8192 and
  // 8192 x 28672 shapes at 8-64 tokens.
  if (M >= 3 && M <= kSkMaxM) {
    const int bn = M <= 16 ? 16 : (M <= 32 ? 32 : 64);
    const int64_t tiles_n = (N + 127) / 128;
    const int num_kt = static_cast<int>(p.Kp / 64);
    int cs = 1, kp = 0;
    if (tiles_n <= 65535 && sk_split(bn, tiles_n, num_kt, kSkMaxCs, &cs, &kp) && tiles_n * cs <= kRefSms) {
      p.path = kSkinny;
      p.bn = bn;
      p.tiles_n = tiles_n;
      p.tiles_m = 1;
      p.sk_cs = cs;
      p.sk_kt_per = kp;
      p.ws_bytes = 0;
      return p;
    }
  }
  p.path = kTc;
  int bn = 16;
  while (bn < M && bn < 256) bn *= 2;
  p.bn = bn;
  p.tiles_n = (N + 127) / 128;
  p.tiles_m = (M + bn - 1) / bn;
  const int64_t tiles = p.tiles_n * p.tiles_m;
  const int num_kt = static_cast<int>(p.Kp / 64);
  // block slots: token tiles of up to 64 run two GEMM blocks per SM
  const int64_t slots = static_cast<int64_t>(kRefSms) * tc_blocks_per_sm(bn);
  int splits = 1;
  if (tiles < slots / 2) {
    int by_sms = static_cast<int>(slots / tiles);
    int by_k = num_kt / 2 > 0 ? num_kt / 2 : 1;
    splits = by_sms < by_k ? by_sms : by_k;
    if (splits < 1) splits = 1;
  }
  p.kt_per_split = (num_kt + splits - 1) / splits;
  p.splits = (num_kt + p.kt_per_split - 1) / p.kt_per_split;
  p.tiles_total = static_cast<int>(tiles < 0x7fffffff ? tiles : 0x7fffffff);
  // Stream-K (a cooperative grid, one block per SM) only for token tiles that
  // run one block per SM; smaller tiles take whole tiles over their 296 slots
  // (a cooperative grid of two blocks per SM was refused at launch).
  if (p.splits == 1 && tc_blocks_per_sm(bn) == 1 && tiles >= kRefSms && tiles * num_kt < 0x7fffffff) {
    const int64_t waves = (tiles + kRefSms - 1) / kRefSms;
    if (tiles * 10 < waves * kRefSms * 9) {  // whole tiles would leave > 10 % of the SMs idle
      p.streamk = 1;
      p.sk_grid = kRefSms;
      p.units = static_cast<int>(tiles * num_kt);
      p.units_per = (p.units + kRefSms - 1) / kRefSms;  // >= num_kt since tiles >= kRefSms
    }
  }
  size_t off = 0;
  p.off_xb = off;
  off = align256(off + static_cast<size_t>(M) * static_cast<size_t>(p.Kp) * 2);
  p.off_sc = off;
  off = align256(off + static_cast<size_t>(M) * 4);
  p.off_acc = off;
  p.off_cnt = off;
  p.off_part = off;
  if (p.splits > 1) {
    off = align256(off + static_cast<size_t>(M) * static_cast<size_t>(N) * 4);
    p.off_cnt = off;
    off = align256(off + static_cast<size_t>(tiles) * 4);
    p.off_part = off;
  }
  if (p.streamk) {
    // int32 partial tile [bn][128] per block, then one flag per block
    off = align256(off + static_cast<size_t>(p.sk_grid) * p.bn * 128 * 4);
    p.off_cnt = off;
    off = align256(off + static_cast<size_t>(p.sk_grid) * 4);
  }
  p.ws_bytes = off;
  return p;
}

struct GemvGrid {
  int grid = 1, rows_per_cta = 1, stage_rows = 1, stage_bytes = 128, nstages = 1, cw = 8;
  int smem = 0;
};

// One block per SM, each a contiguous run of rows.  Single-token blocks with
// much work get 16 consumer warps; the others 8, which leaves room for a
// block of the next kernel to start alongside under launch overlap.
inline GemvGrid gemv_grid(const Plan &p, int sms) {
  GemvGrid g;
  const int64_t rpc = (p.N + sms - 1) / sms;
  g.rows_per_cta = static_cast<int>(rpc);
  g.grid = static_cast<int>((p.N + rpc - 1) / rpc);
  int64_t sr = kGemvStageBytes / p.row_bytes;
  if (p.split_log2 > 0 && sr > kGemvMaxSplitRows) sr = kGemvMaxSplitRows;
  if (sr < 1) sr = 1;
  if (sr > rpc) sr = rpc;
  g.stage_rows = static_cast<int>(sr);
  g.stage_bytes = static_cast<int>(((sr * p.row_bytes) + 127) / 128 * 128);
  const int64_t iters = (rpc + sr - 1) / sr;
  const int64_t codes = p.M * p.Kp;
  int64_t S = iters < kGemvMaxStages ? iters : kGemvMaxStages;
  while (S > 1 && kGemvSmemFixed + S * g.stage_bytes + codes > kSmemMax) --S;
  g.nstages = static_cast<int>(S);
  g.smem = static_cast<int>(kGemvSmemFixed + S * g.stage_bytes + codes);
  g.cw = (p.mt == 1 && rpc * p.row_bytes >= 64 * 1024) ? 16 : 8;
  return g;
}

}  // namespace plan
}  // namespace bl
