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
constexpr int kGemvThreads = 256;        // consumer threads of the GEMV kernel
constexpr int kGemvStageBytes = 32 * 1024;

inline int64_t row_bytes(int64_t K) { return ((K + 63) / 64) * 16; }

inline size_t align256(size_t v) { return (v + 255) & ~static_cast<size_t>(255); }

struct Plan {
  int path = kGemv;
  int64_t M = 0, N = 0, K = 0, Kp = 0, row_bytes = 0;
  // GEMV: tokens per thread (1, 2 or 4), words per thread, log2 threads per row
  int mt = 1, wpt = 1, tpr_log2 = 0;
  // tensor-core GEMM
  int bn = 0;
  int64_t tiles_n = 0, tiles_m = 0;
  int tiles_total = 0;
  int splits = 1, kt_per_split = 0;
  // workspace (bytes, 256-aligned offsets)
  size_t off_xb = 0, off_sc = 0, off_acc = 0, off_cnt = 0, ws_bytes = 0;
};

inline int wpt_max(int mt) { return mt == 1 ? 8 : (mt == 2 ? 4 : 2); }

inline Plan make(int64_t M, int64_t N, int64_t K) {
  Plan p;
  p.M = M;
  p.N = N;
  p.K = K;
  p.row_bytes = row_bytes(K);
  p.Kp = p.row_bytes * 4;
  const int64_t words = p.row_bytes / 4;
  if (M <= 4) {
    p.mt = M == 1 ? 1 : (M == 2 ? 2 : 4);
    const int wm = wpt_max(p.mt);
    int best = -1;
    int64_t best_waste = 0;
    for (int lg = 0; lg <= 8; ++lg) {
      const int64_t tpr = int64_t(1) << lg;
      const int64_t w = (words + tpr - 1) / tpr;
      if (w > wm) continue;
      const int64_t waste = tpr * w - words;
      if (best < 0 || waste < best_waste) {
        best = lg;
        best_waste = waste;
      }
    }
    if (best >= 0) {
      p.path = kGemv;
      p.tpr_log2 = best;
      p.wpt = static_cast<int>((words + (int64_t(1) << best) - 1) >> best);
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
  int grid = 1, rows_per_cta = 1, stage_rows = 1;
};

inline GemvGrid gemv_grid(const Plan &p, int sms) {
  GemvGrid g;
  const int64_t rpi = kGemvThreads >> p.tpr_log2;
  int64_t want = (p.N + rpi - 1) / rpi;
  if (want > sms) want = sms;
  if (want < 1) want = 1;
  const int64_t rpc = (p.N + want - 1) / want;
  g.rows_per_cta = static_cast<int>(rpc);
  g.grid = static_cast<int>((p.N + rpc - 1) / rpc);
  int64_t sr = kGemvStageBytes / p.row_bytes;
  if (sr < 1) sr = 1;
  if (sr >= rpi) sr -= sr % rpi;
  if (sr > rpc) sr = rpc;
  g.stage_rows = static_cast<int>(sr);
  return g;
}

}  // namespace plan
}  // namespace bl
