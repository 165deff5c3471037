// Launch-plan invariants of the BitLinear library, checked on the host over
// a grid of shapes: every GEMV plan covers each row with at most the block's
// warps, its stages fit their buffers and shared memory, its grid covers N
// exactly once; every tensor-core plan covers M, N and all k tiles; every
// few-token plan gives each block of a cluster at least one k tile, fits its
// operands in shared memory and holds the split-K sums it receives, and its
// clusters fit one wave of blocks; GEMM plans count two blocks per SM for
// token tiles of up to 64 and use stream-K only at one block per SM.
#include <cstdio>
#include <cstdlib>
#include <initializer_list>
#include "bl_plan.h"
using namespace bl::plan;
int main() {
  long checked = 0, gemv = 0, tc = 0, sk = 0, streamk = 0;
  const int sms = 148;
  for (long M = 1; M <= 300; M += (M < 16 ? 1 : 37))
    for (long K : {1L, 15L, 16L, 63L, 64L, 65L, 100L, 333L, 512L, 1000L, 2560L, 4096L, 6912L, 8192L, 9000L, 16384L, 28672L, 32768L, 65536L, 131072L})
      for (long N : {1L, 7L, 128L, 129L, 256L, 300L, 513L, 2560L, 3840L, 6912L, 8192L, 28672L, 40960L}) {
        Plan p = make(M, N, K);
        ++checked;
        // the GEMV takes exactly the calls the header documents for launch
        // overlap mode 2
        const bool want_gemv = (M == 1 && K <= 65536) || (M == 2 && K <= 32768) || ((M == 3 || M == 4) && K <= 16384);
        if ((p.path == kGemv) != want_gemv) { printf("BAD route M=%ld N=%ld K=%ld\n", M, N, K); return 1; }
        if (p.path == kGemv) {
          ++gemv;
          const int G = 1 << p.split_log2;
          const long units = p.row_bytes / 8;
          GemvGrid g = gemv_grid(p, sms);
          bool ok = M <= 4 && G <= g.cw && (g.cw >> p.split_log2) >= 1 &&
                    (long)p.chunk * G >= units && p.upt * 32 >= p.chunk && p.upt >= 1 &&
                    p.upt <= upt_max(p.mt) && (g.cw == 8 || (g.cw == 16 && p.mt == 1));
          ok = ok && g.grid >= 1 && (long)g.grid * g.rows_per_cta >= N && (long)(g.grid - 1) * g.rows_per_cta < N;
          ok = ok && g.stage_rows >= 1 && g.stage_rows <= g.rows_per_cta && g.nstages >= 1 && g.nstages <= kGemvMaxStages;
          ok = ok && (long)g.stage_rows * p.row_bytes <= g.stage_bytes && g.stage_bytes % 128 == 0;
          ok = ok && ((long)g.stage_rows * p.row_bytes <= kGemvStageBytes || g.stage_rows == 1);
          ok = ok && (p.split_log2 == 0 || g.stage_rows <= kGemvMaxSplitRows);
          ok = ok && g.smem <= kSmemMax &&
               g.smem == kGemvSmemFixed + g.nstages * g.stage_bytes + (int)(M * p.Kp);
          if (!ok) { printf("BAD gemv M=%ld N=%ld K=%ld G=%d upt=%d chunk=%d\n", M, N, K, G, p.upt, p.chunk); return 1; }
        } else if (p.path == kSkinny) {
          ++sk;
          const long nkt = p.Kp / 64;
          bool ok = M >= 3 && M <= kSkMaxM && (p.bn == 16 || p.bn == 32 || p.bn == 64) && p.bn >= M &&
                    p.tiles_n * 128 >= N && (p.tiles_n - 1) * 128 < N && p.ws_bytes == 0 &&
                    p.tiles_n * p.sk_cs <= kRefSms;
          ok = ok && p.sk_cs >= 1 && p.sk_cs <= kSkMaxCs && p.sk_kt_per >= 1 &&
               (long)p.sk_cs * p.sk_kt_per >= nkt && (long)(p.sk_cs - 1) * p.sk_kt_per < nkt;
          // every smaller cluster the launch may pick instead keeps the same properties
          for (int c = p.sk_cs; ok && c >= 1; --c) {
            const int kp = (int)((nkt + c - 1) / c), cc = (int)((nkt + kp - 1) / kp);
            if (sk_ring(p.bn, kp, cc) == 0) continue;
            const long last = nkt - (long)(cc - 1) * kp;
            ok = ok && last >= 1 && last <= kp && cc <= kSkMaxCs;
            ok = ok && sk_launch_smem(p.bn, kp, cc) <= kSmemMax && sk_launch_smem(p.bn, kp, cc) >= kSkSmemFloor;
            ok = ok && sk_ring(p.bn, kp, cc) >= 2 * sk_lanes(p.bn) && sk_ring(p.bn, kp, cc) <= kSkMaxWs && sk_ring(p.bn, kp, cc) % sk_lanes(p.bn) == 0;
            ok = ok && (cc == 1 || sk_red_bytes(p.bn, cc) >= (long)cc * ((M + cc - 1) / cc) * 512);
          }
          if (!ok) { printf("BAD skinny M=%ld N=%ld K=%ld cs=%d kp=%d\n", M, N, K, p.sk_cs, p.sk_kt_per); return 1; }
        } else {
          ++tc;
          streamk += p.streamk;
          bool ok = p.bn >= 16 && p.bn <= 256 && p.splits >= 1 && p.kt_per_split >= 1 &&
                    (long)p.splits * p.kt_per_split >= p.Kp / 64 && (long)(p.splits - 1) * p.kt_per_split < p.Kp / 64 &&
                    p.tiles_n * 128 >= N && p.tiles_m * p.bn >= M;
          if (p.streamk) {
            // every block's share spans at least one whole tile (so a tile is
            // split between at most two neighbouring blocks) and the shares cover
            // every unit once (trailing blocks may get none); the workspace holds
            // one partial tile and one flag per block
            const long nkt = p.Kp / 64;
            ok = ok && p.splits == 1 && tc_blocks_per_sm(p.bn) == 1 && p.sk_grid == kRefSms && p.units == (long)p.tiles_total * nkt &&
                 p.units_per >= nkt && (long)p.units_per * p.sk_grid >= p.units &&
                 p.off_cnt >= p.off_part + (size_t)p.sk_grid * p.bn * 128 * 4 &&
                 p.ws_bytes >= p.off_cnt + (size_t)p.sk_grid * 4;
          }
          if (!ok) { printf("BAD tc M=%ld N=%ld K=%ld\n", M, N, K); return 1; }
        }
      }
  printf("ok: %ld plans (%ld gemv, %ld tensor-core of which %ld stream-K, %ld few-token)\n", checked, gemv, tc, streamk, sk);
  // the specific shapes of the tests and bench
  for (long M : {1L, 3L, 8L}) for (long K : {2560L, 6912L, 8192L, 28672L}) {
    Plan p = make(M, 2560, K);
    printf("M=%ld K=%ld path=%s G=%d upt=%d chunk=%d\n", M, K,
           p.path == kGemv ? "gemv" : (p.path == kSkinny ? "skinny" : "tc"), 1 << p.split_log2, p.upt, p.chunk);
  }
  return 0;
}
