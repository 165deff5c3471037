// Host-side planning for the BitLinear forward: which kernel runs for a given
// (M, N, K), its tiling, and the workspace layout.  Pure integer logic, so
// the workspace size a caller queries is the one the call uses.
#pragma once

#include <cstddef>
#include <cstdint>

namespace bl {
namespace plan {

enum Path { kGemv = 0, kTc = 1 };

// Reference SM count used for split-K decisions (B300: 148 SMs).  A fixed
// value keeps workspace sizes independent of the device.
constexpr int kRefSms = 148;
constexpr int kGemvStageBytes = 32 * 1024;   // upper bound of one GEMV ring stage
constexpr int kGemvMaxStages = 6;
constexpr int kGemvMaxSplitRows = 32;
constexpr int kGemvSmemFixed = 8 * 1024;
constexpr int kSmemMax = 227 * 1024;

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
  // workspace (bytes, 256-aligned offsets)
  size_t off_xb = 0, off_sc = 0, off_acc = 0, off_cnt = 0, ws_bytes = 0;
};

// Units per lane so the activation slice stays within 64 registers
// (8 registers per unit and token).
inline int upt_max(int mt) { return mt == 1 ? 8 : (mt == 2 ? 4 : (mt == 4 ? 2 : 1)); }

inline Plan make(int64_t M, int64_t N, int64_t K) {
  Plan p;
  p.M = M;
  p.N = N;
  p.K = K;
  p.row_bytes = row_bytes(K);
  p.Kp = p.row_bytes * 4;
  const int64_t units = p.row_bytes / 8;
  if (M <= 8) {
    p.mt = M == 1 ? 1 : (M == 2 ? 2 : (M <= 4 ? 4 : 8));
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
  p.path = kTc;
  int bn = 16;
  while (bn < M && bn < 256) bn *= 2;
  p.bn = bn;
  p.tiles_n = (N + 127) / 128;
  p.tiles_m = (M + bn - 1) / bn;
  const int64_t tiles = p.tiles_n * p.tiles_m;
  const int num_kt = static_cast<int>(p.Kp / 64);
  int splits = 1;
  if (tiles < kRefSms / 2) {
    int by_sms = static_cast<int>(kRefSms / tiles);
    int by_k = num_kt / 2 > 0 ? num_kt / 2 : 1;
    splits = by_sms < by_k ? by_sms : by_k;
    if (splits < 1) splits = 1;
  }
  p.kt_per_split = (num_kt + splits - 1) / splits;
  p.splits = (num_kt + p.kt_per_split - 1) / p.kt_per_split;
  p.tiles_total = static_cast<int>(tiles < 0x7fffffff ? tiles : 0x7fffffff);
  size_t off = 0;
  p.off_xb = off;
  off = align256(off + static_cast<size_t>(M) * static_cast<size_t>(p.Kp) * 2);
  p.off_sc = off;
  off = align256(off + static_cast<size_t>(M) * 4);
  p.off_acc = off;
  p.off_cnt = off;
  if (p.splits > 1) {
    off = align256(off + static_cast<size_t>(M) * static_cast<size_t>(N) * 4);
    p.off_cnt = off;
    off = align256(off + static_cast<size_t>(tiles) * 4);
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
