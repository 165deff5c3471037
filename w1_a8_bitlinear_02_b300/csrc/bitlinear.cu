// C ABI of the BitLinear W1.58A8 forward (see include/bitlinear.h).
// Host side: argument checks, path planning, TMA descriptors, launches.
#include "bitlinear.h"

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <set>
#include <tuple>
#include <utility>
#include <vector>

#include "bl_chain.cuh"
#include "bl_gemm_tc.cuh"
#include "bl_gemv.cuh"
#include "bl_pack_quant.cuh"
#include "bl_plan.h"
#include "bl_ptx.cuh"
#include "bl_skinny.cuh"

// Scratch memory for bitlinear_forward_noalloc: a fixed array in the
// library's own device memory, so that entry point never allocates.  Every GPU
// that loads the library holds these bytes until the process exits.
constexpr size_t kNoAllocScratchBytes = size_t(8) << 20;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

namespace {

using namespace bl;

std::atomic<int> g_overlap{0};

constexpr int64_t kMaxK = 131072;
constexpr int64_t kMaxDim = 2147483647;

// ------------------------------------------------------------ device checks
struct DevState {
  bool probed = false;
  bool supported = false;
  int sms = 0;
  std::set<const void *> smem_set;  // kernels whose dynamic-smem limit was raised
};
constexpr int kMaxDevices = 64;  // device ordinals this library keeps state for
std::mutex g_mu;
DevState g_dev[kMaxDevices];

bl_status current_device(int *dev, int *sms) {
  int d = 0;
  if (cudaGetDevice(&d) != cudaSuccess) {
    cudaGetLastError();
    return BL_ERR_CUDA;
  }
  if (d < 0 || d >= kMaxDevices) return BL_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lk(g_mu);
  DevState &st = g_dev[d];
  if (!st.probed) {
    int major = 0, minor = 0, n = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, d) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, d) != cudaSuccess ||
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, d) != cudaSuccess) {
      cudaGetLastError();
      return BL_ERR_CUDA;
    }
    st.probed = true;
    st.supported = (major == 10 && minor == 3);
    st.sms = n;
  }
  if (!st.supported) return BL_ERR_UNSUPPORTED;
  *dev = d;
  if (sms) *sms = st.sms;
  return BL_OK;
}

bl_status ensure_smem(int dev, const void *func, int bytes) {
  std::lock_guard<std::mutex> lk(g_mu);
  DevState &st = g_dev[dev];
  if (st.smem_set.count(func)) return BL_OK;
  if (cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess) {
    cudaGetLastError();
    return BL_ERR_CUDA;
  }
  st.smem_set.insert(func);
  return BL_OK;
}

// A launch the runtime refused: cleared and reported as BL_ERR_CUDA; with
// BITLINEAR_DEBUG set in the environment the CUDA error text goes to stderr.
bl_status launch_failed(const char *what) {
  const cudaError_t e = cudaGetLastError();
  static const bool dbg = std::getenv("BITLINEAR_DEBUG") != nullptr;
  if (dbg) std::fprintf(stderr, "bitlinear: %s: %s\n", what, cudaGetErrorString(e));
  return BL_ERR_CUDA;
}

template <typename... KArgs, typename... Args>
bl_status launch(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                 bool overlap, Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  if (overlap) {
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  if (cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...) != cudaSuccess) return launch_failed("launch");
  return BL_OK;
}

// ------------------------------------------------------------ TMA descriptors
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    else
      cudaGetLastError();
  });
  return fn;
}

// bf16 activations [rows, ld] (k innermost), box 64 x box_rows, 128-byte swizzle.
bool make_map_x(CUtensorMap *m, const void *ptr, int64_t rows, int64_t ld, int box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(ld), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld * 2)};
  cuuint32_t box[2] = {64u, static_cast<cuuint32_t>(box_rows)};
  cuuint32_t es[2] = {1u, 1u};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(ptr), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// packed weights [N, row_bytes] bytes, box 16 bytes x 128 rows, no swizzle.
bool make_map_w(CUtensorMap *m, const void *ptr, int64_t N, int64_t row_bytes) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(row_bytes), static_cast<cuuint64_t>(N)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(row_bytes)};
  cuuint32_t box[2] = {16u, static_cast<cuuint32_t>(tc::kBM)};
  cuuint32_t es[2] = {1u, 1u};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(ptr), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

bl_status check_dims(int64_t M, int64_t N, int64_t K) {
  if (M < 1 || M > kMaxDim || N < 1 || N > kMaxDim || K < 1 || K > kMaxK) return BL_ERR_SHAPE;
  return BL_OK;
}

// The launch grids a plan needs must exist: the tensor-core GEMM puts token
// tiles and K splits on grid dimensions y and z (at most 65535 each), the
// few-token kernel its row tiles on y.  Checked before anything is enqueued.
bl_status check_grid(const plan::Plan &pl) {
  if (pl.path == plan::kTc && (pl.tiles_m > 65535 || pl.splits > 65535 || pl.tiles_n > 0x7fffffff))
    return BL_ERR_SHAPE;
  if (pl.path == plan::kSkinny && pl.tiles_n > 65535) return BL_ERR_SHAPE;
  return BL_OK;
}

// ------------------------------------------------------------ GEMV dispatch
template <int MT, int XM, bool OUT_I32, int CW>
void *gemv_func_upt(int upt) {
#define BL_G(U) reinterpret_cast<void *>(&gemv::gemv_kernel<MT, U, XM, OUT_I32, CW>)
  if (upt == 1) return BL_G(1);
  if constexpr (MT <= 4) {
    if (upt == 2) return BL_G(2);
  }
  if constexpr (MT <= 2) {
    if (upt == 3) return BL_G(3);
    if (upt == 4) return BL_G(4);
  }
  if constexpr (MT == 1) {
    if (upt == 5) return BL_G(5);
    if (upt == 6) return BL_G(6);
    if (upt == 7) return BL_G(7);
    if (upt == 8) return BL_G(8);
  }
#undef BL_G
  return nullptr;
}

template <int XM, bool OUT_I32, int CW>
void *gemv_func_m(int mt, int upt) {
  if (mt == 1) return gemv_func_upt<1, XM, OUT_I32, CW>(upt);
  if constexpr (CW == 16) {
    return nullptr;  // 16 consumer warps only for one token
  } else {
    if (mt == 2) return gemv_func_upt<2, XM, OUT_I32, CW>(upt);
    if (mt == 4) return gemv_func_upt<4, XM, OUT_I32, CW>(upt);
    return gemv_func_upt<8, XM, OUT_I32, CW>(upt);
  }
}

template <int CW>
void *gemv_func(int xm, bool out_i32, int mt, int upt) {
  if (out_i32) return gemv_func_m<gemv::kXInt8, true, CW>(mt, upt);
  if (xm == gemv::kXF32) return gemv_func_m<gemv::kXF32, false, CW>(mt, upt);
  if (xm == gemv::kXBF16) return gemv_func_m<gemv::kXBF16, false, CW>(mt, upt);
  return gemv_func_m<gemv::kXInt8, false, CW>(mt, upt);
}

bl_status run_gemv(const plan::Plan &pl, int dev, int sms, int xm, int act, bool out_i32, const uint8_t *packed,
                   const float *gamma, const void *x, const int8_t *xq, const float *scale, const OutSpec &out,
                   int32_t *acc, cudaStream_t st) {
  const plan::GemvGrid g = plan::gemv_grid(pl, sms);
  void *f = g.cw == 16 ? gemv_func<16>(xm, out_i32, pl.mt, pl.upt) : gemv_func<8>(xm, out_i32, pl.mt, pl.upt);
  if (!f) return BL_ERR_UNSUPPORTED;
  bl_status s = ensure_smem(dev, f, plan::kSmemMax);
  if (s != BL_OK) return s;
  gemv::Params p{};
  p.packed = packed;
  p.gamma = gamma;
  p.x = x;
  p.xq = xq;
  p.scale = scale;
  p.out = out;
  p.acc = acc;
  p.N = pl.N;
  p.K = static_cast<int>(pl.K);
  p.kp = static_cast<int>(pl.Kp);
  p.units = static_cast<int>(pl.row_bytes / 8);
  p.row_bytes = static_cast<int>(pl.row_bytes);
  p.M = static_cast<int>(pl.M);
  p.rows_per_cta = g.rows_per_cta;
  p.stage_rows = g.stage_rows;
  p.stage_bytes = g.stage_bytes;
  p.nstages = g.nstages;
  p.split_log2 = pl.split_log2;
  p.chunk = pl.chunk;
  const int ov = g_overlap.load();
  p.wait_prior = ov == 2 ? 0 : 1;
  p.act = act;
  return launch(reinterpret_cast<void (*)(gemv::Params)>(f), dim3(g.grid), dim3((g.cw + 1) * 32), g.smem,
                st, ov != 0, p);
}

// ------------------------------------------------------------ tensor-core dispatch
static_assert(plan::tc_blocks_per_sm(16) == tc::blocks_per_sm(16) && plan::tc_blocks_per_sm(32) == tc::blocks_per_sm(32) &&
                  plan::tc_blocks_per_sm(64) == tc::blocks_per_sm(64) &&
                  plan::tc_blocks_per_sm(128) == tc::blocks_per_sm(128) &&
                  plan::tc_blocks_per_sm(256) == tc::blocks_per_sm(256),
              "planner and GEMM kernel agree on blocks per SM");
template <int BN, bool OUT_I32, bool GROUPED>
bl_status run_tc_bn(const plan::Plan &pl, int dev, const CUtensorMap &mx, const CUtensorMap &mw,
                    const tc::Params &p, cudaStream_t st) {
  auto *f = &tc::tc_gemm_kernel<BN, OUT_I32, GROUPED>;
  constexpr int smem = tc::Cfg<BN>::kSmemBytes;
  bl_status s = ensure_smem(dev, reinterpret_cast<const void *>(f), smem);
  if (s != BL_OK) return s;
  if (p.streamk) {
    // One block per SM, all resident at once (a block may wait for its
    // neighbour's partial): a cooperative launch, ordered after the previous
    // kernel (which zeroed the flags) without launch overlap.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(pl.sk_grid));
    cfg.blockDim = dim3(tc::kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, f, mx, mw, p) != cudaSuccess) {
      cudaGetLastError();
      return BL_ERR_CUDA;
    }
    return BL_OK;
  }
  dim3 grid(static_cast<unsigned>(pl.tiles_n), static_cast<unsigned>(pl.tiles_m),
            static_cast<unsigned>(pl.splits));
  return launch(f, grid, dim3(tc::kThreads), smem, st, g_overlap.load() != 0, mx, mw, p);
}

template <bool OUT_I32, bool GROUPED>
bl_status run_tc_g(const plan::Plan &pl, int dev, const CUtensorMap &mx, const CUtensorMap &mw,
                   const tc::Params &p, cudaStream_t st) {
  switch (pl.bn) {
    case 16: return run_tc_bn<16, OUT_I32, GROUPED>(pl, dev, mx, mw, p, st);
    case 32: return run_tc_bn<32, OUT_I32, GROUPED>(pl, dev, mx, mw, p, st);
    case 64: return run_tc_bn<64, OUT_I32, GROUPED>(pl, dev, mx, mw, p, st);
    case 128: return run_tc_bn<128, OUT_I32, GROUPED>(pl, dev, mx, mw, p, st);
    case 256: return run_tc_bn<256, OUT_I32, GROUPED>(pl, dev, mx, mw, p, st);
    default: return BL_ERR_UNSUPPORTED;
  }
}

template <bool OUT_I32>
bl_status run_tc(const plan::Plan &pl, int dev, const CUtensorMap &mx, const CUtensorMap &mw,
                 const tc::Params &p, cudaStream_t st) {
  if (!OUT_I32 && p.out.gvec != nullptr) return run_tc_g<OUT_I32, true>(pl, dev, mx, mw, p, st);
  return run_tc_g<OUT_I32, false>(pl, dev, mx, mw, p, st);
}

// ------------------------------------------------------------ few-token dispatch
template <int XM, bool OUT_I32>
void *sk_func_bn(int bn) {
  if (bn == 16) return reinterpret_cast<void *>(&sk::skinny_kernel<16, XM, OUT_I32>);
  if (bn == 32) return reinterpret_cast<void *>(&sk::skinny_kernel<32, XM, OUT_I32>);
  if (bn == 64) return reinterpret_cast<void *>(&sk::skinny_kernel<64, XM, OUT_I32>);
  return nullptr;
}

void *sk_func(int bn, int xm, bool out_i32) {
  if (out_i32) return sk_func_bn<sk::kXInt8, true>(bn);
  if (xm == gemv::kXF32) return sk_func_bn<sk::kXF32, false>(bn);
  if (xm == gemv::kXBF16) return sk_func_bn<sk::kXBF16, false>(bn);
  return sk_func_bn<sk::kXInt8, false>(bn);
}

// Clusters of `cs` blocks of kernel f (with `smem` bytes each) that the device
// can hold at once; cached.
std::map<std::tuple<int, const void *, int, int>, int> g_cluster_cap;

int sk_threads(int bn) { return 32 * (1 + 5 * sk::lanes_for(bn)); }

int cluster_capacity(int dev, const void *f, int cs, int smem, int threads) {
  const auto key = std::make_tuple(dev, f, cs, smem);
  {
    std::lock_guard<std::mutex> lk(g_mu);
    auto it = g_cluster_cap.find(key);
    if (it != g_cluster_cap.end()) return it->second;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(cs), 1, 1);
  cfg.blockDim = dim3(static_cast<unsigned>(threads));
  cfg.dynamicSmemBytes = static_cast<size_t>(smem);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(cs);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, f, &cfg) != cudaSuccess) {
    cudaGetLastError();
    n = 0;
  }
  std::lock_guard<std::mutex> lk(g_mu);
  g_cluster_cap[key] = n;
  return n;
}

bl_status run_skinny(const plan::Plan &pl, int dev, int xm, int act, bool out_i32, const uint8_t *packed,
                     const float *gamma, const void *x, const int8_t *xq, const float *scale, const OutSpec &out,
                     int32_t *acc, cudaStream_t st) {
  void *f = sk_func(pl.bn, xm, out_i32);
  if (!f) return BL_ERR_UNSUPPORTED;
  bl_status s = ensure_smem(dev, f, plan::kSmemMax);
  if (s != BL_OK) return s;
  const int num_kt = static_cast<int>(pl.Kp / 64);
  // The plan's cluster size assumes every SM can host a block of a cluster;
  // a smaller cluster wins when fewer clusters of the planned size fit at
  // once.  Cost of a choice: waves x (k tiles per block + fixed cost).
  int best_cs = pl.sk_cs, best_kp = pl.sk_kt_per;
  double best_cost = 0.0;
  for (int c = pl.sk_cs; c >= 1; --c) {
    const int kp = (num_kt + c - 1) / c;
    const int cc = (num_kt + kp - 1) / kp;
    if (plan::sk_ring(pl.bn, kp, cc) == 0) continue;
    const int cap = cluster_capacity(dev, f, cc, plan::sk_launch_smem(pl.bn, kp, cc), sk_threads(pl.bn));
    if (cap <= 0) continue;
    const double waves = static_cast<double>((pl.tiles_n + cap - 1) / cap);
    const double cost = waves * (kp + 24.0);
    if (best_cost == 0.0 || cost < best_cost) {
      best_cost = cost;
      best_cs = cc;
      best_kp = kp;
    }
  }
  CUtensorMap mw, mx;
  std::memset(&mx, 0, sizeof(mx));
  if (!make_map_w(&mw, packed, pl.N, pl.row_bytes)) return BL_ERR_CUDA;
  // bf16 rows with 16-byte aligned starts come by TMA into the B operand
  const bool x_tma = !out_i32 && xm == gemv::kXBF16 && pl.K % 8 == 0 && aligned(x, 16);
  if (x_tma && !make_map_x(&mx, x, pl.M, pl.K, pl.bn)) return BL_ERR_CUDA;
  sk::Params p{};
  p.x = out_i32 || xm == gemv::kXInt8 ? static_cast<const void *>(xq) : x;
  p.scale = scale;
  p.gamma = gamma;
  p.out = out;
  p.acc = acc;
  p.M = static_cast<int>(pl.M);
  p.N = static_cast<int>(pl.N);
  p.K = static_cast<int>(pl.K);
  p.num_kt = num_kt;
  p.kt_per = best_kp;
  p.cs = best_cs;
  p.ws = plan::sk_ring(pl.bn, best_kp, best_cs);
  p.x_tma = x_tma ? 1 : 0;
  p.act = act;
  const int smem = plan::sk_launch_smem(pl.bn, best_kp, best_cs);

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(best_cs), static_cast<unsigned>(pl.tiles_n), 1);
  cfg.blockDim = dim3(static_cast<unsigned>(sk_threads(pl.bn)));
  cfg.dynamicSmemBytes = static_cast<size_t>(smem);
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(best_cs);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  int na = 1;
  if (g_overlap.load() != 0) {
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    na = 2;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  if (cudaLaunchKernelEx(&cfg, reinterpret_cast<void (*)(CUtensorMap, CUtensorMap, sk::Params)>(f), mw, mx,
                         p) !=
      cudaSuccess) {
    cudaGetLastError();
    return BL_ERR_CUDA;
  }
  return BL_OK;
}

// Shared body of forward / forward_q / matmul_i32 on the tensor-core path.
// xm: activation source (f32 / bf16 to be quantised, or int8 codes).
bl_status forward_tc(const plan::Plan &pl, int dev, int xm, int act, bool out_i32, const uint8_t *packed,
                     const float *gamma, const void *x, const int8_t *xq, const float *scale, const OutSpec &out,
                     int32_t *acc, void *ws, size_t ws_bytes, cudaStream_t st) {
  if (ws == nullptr || ws_bytes < pl.ws_bytes) return BL_ERR_WORKSPACE;
  if (!aligned(ws, 256)) return BL_ERR_ALIGN;
  uint8_t *w = static_cast<uint8_t *>(ws);
  auto *xb = reinterpret_cast<__nv_bfloat16 *>(w + pl.off_xb);
  float *sc = reinterpret_cast<float *>(w + pl.off_sc);
  int32_t *wacc = reinterpret_cast<int32_t *>(w + pl.off_acc);
  unsigned *wcnt = reinterpret_cast<unsigned *>(w + pl.off_cnt);
  const bool overlap = g_overlap.load() != 0;

  CUtensorMap mx, mw;
  if (!make_map_x(&mx, xb, pl.M, pl.Kp, pl.bn) || !make_map_w(&mw, packed, pl.N, pl.row_bytes))
    return BL_ERR_CUDA;

  // Stream-K needs every block resident at once: one block per SM of a
  // device with at least the planned number of SMs; otherwise whole tiles.
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    cudaGetLastError();
    return BL_ERR_CUDA;
  }
  const bool streamk = pl.streamk && sms * tc::blocks_per_sm(pl.bn) >= pl.sk_grid;

  // 1) activations -> bf16 codes (+ scales), zeroing the split-K accumulators
  //    or the stream-K flags
  const bool zero_acc = pl.splits > 1;
  int32_t *zrows = zero_acc ? (out_i32 ? acc : wacc) : nullptr;
  unsigned *zcnt = (zero_acc && !out_i32) || streamk ? wcnt : nullptr;
  const int ncnt = streamk ? pl.sk_grid : pl.tiles_total;
  bl_status s;
  const dim3 qgrid(static_cast<unsigned>(pl.M));
  const float *use_scale = scale;
  if (xm == gemv::kXInt8) {
    s = launch(&codes_to_bf16_kernel, qgrid, dim3(256), 0, st, overlap, xq, pl.K, pl.Kp, xb, zrows,
               pl.N, zcnt, ncnt);
  } else {
    use_scale = sc;
    // one pass with the rows in registers, several rows a block, where the
    // shape allows (measured: 2048 x 2560 forward 70.5 -> 69.5 us; at one
    // 6912-long row a block it gained nothing, so longer rows keep the
    // two-pass kernel)
    const int tpr = pl.K <= 2048 ? 64 : (pl.K <= 4096 ? 128 : 0);
    const bool fast = tpr > 0 && pl.K % 8 == 0 && aligned(x, 16) && aligned(xb, 16) && pl.Kp % 8 == 0;
    if (fast) {
      const dim3 fgrid(static_cast<unsigned>((pl.M + 256 / tpr - 1) / (256 / tpr)));
      if (xm == gemv::kXF32) {
        const float *xf = static_cast<const float *>(x);
        s = tpr == 64 ? launch(&quant_rows_bf16_kernel<float, 64>, fgrid, dim3(256), 0, st, overlap, xf, pl.M, pl.K,
                               pl.Kp, xb, sc, zrows, pl.N, zcnt, ncnt, act)
                      : launch(&quant_rows_bf16_kernel<float, 128>, fgrid, dim3(256), 0, st, overlap, xf, pl.M,
                               pl.K, pl.Kp, xb, sc, zrows, pl.N, zcnt, ncnt, act);
      } else {
        const __nv_bfloat16 *xh = static_cast<const __nv_bfloat16 *>(x);
        s = tpr == 64 ? launch(&quant_rows_bf16_kernel<__nv_bfloat16, 64>, fgrid, dim3(256), 0, st, overlap, xh, pl.M,
                               pl.K, pl.Kp, xb, sc, zrows, pl.N, zcnt, ncnt, act)
                      : launch(&quant_rows_bf16_kernel<__nv_bfloat16, 128>, fgrid, dim3(256), 0, st, overlap, xh,
                               pl.M, pl.K, pl.Kp, xb, sc, zrows, pl.N, zcnt, ncnt, act);
      }
    } else if (xm == gemv::kXF32)
      s = launch(&quant_act_kernel<float, true, false>, qgrid, dim3(256), 0, st, overlap,
                 static_cast<const float *>(x), pl.K, pl.Kp, static_cast<const float *>(nullptr), 0.0f,
                 static_cast<int8_t *>(nullptr), xb, sc, zrows, pl.N, zcnt, ncnt, act);
    else
      s = launch(&quant_act_kernel<__nv_bfloat16, true, false>, qgrid, dim3(256), 0, st, overlap,
                 static_cast<const __nv_bfloat16 *>(x), pl.K, pl.Kp, static_cast<const float *>(nullptr),
                 0.0f, static_cast<int8_t *>(nullptr), xb, sc, zrows, pl.N, zcnt, ncnt, act);
  }
  if (s != BL_OK) return s;

  // 2) the contraction
  tc::Params p{};
  p.N = static_cast<int>(pl.N);
  p.M = static_cast<int>(pl.M);
  p.num_kt = static_cast<int>(pl.Kp / tc::kBK);
  p.kt_per_split = pl.kt_per_split;
  p.splits = pl.splits;
  p.gamma = gamma;
  p.scale = use_scale;
  p.out = out;
  p.acc_out = acc;
  p.ws_acc = wacc;
  p.ws_cnt = wcnt;
  p.streamk = streamk ? 1 : 0;
  p.tiles_n = static_cast<int>(pl.tiles_n);
  p.units = pl.units;
  p.units_per = pl.units_per;
  p.ws_part = reinterpret_cast<int32_t *>(w + pl.off_part);
  p.ws_flag = wcnt;
  if (out_i32) return run_tc<true>(pl, dev, mx, mw, p, st);
  return run_tc<false>(pl, dev, mx, mw, p, st);
}

OutSpec out_f32(float *y) { return OutSpec{y, nullptr, 0}; }

// y: fp32 [M, N] unless out.bf16; out.res: optional residual of y's dtype.
bl_status forward_common(const uint8_t *packed, const float *gamma, int64_t N, int64_t K, int xm, int act,
                         const void *x, const int8_t *xq, const float *scale, int64_t M, OutSpec out,
                         int32_t *acc, void *ws, size_t ws_bytes, void *stream) {
  const bool out_i32 = acc != nullptr;
  if (packed == nullptr || (!out_i32 && (gamma == nullptr || out.y == nullptr)))
    return BL_ERR_NULL;
  if (xm == gemv::kXInt8 ? xq == nullptr : x == nullptr) return BL_ERR_NULL;
  if (xm == gemv::kXInt8 && !out_i32 && scale == nullptr) return BL_ERR_NULL;
  bl_status s = check_dims(M, N, K);
  if (s != BL_OK) return s;
  if (!aligned(packed, 16)) return BL_ERR_ALIGN;
  if (N > 0x7fffffffLL / 1 || static_cast<double>(M) * static_cast<double>(N) > 9.0e15)
    return BL_ERR_SHAPE;
  const plan::Plan pl = plan::make(M, N, K);
  if (pl.path == plan::kTc && (M > 0x7fffffff || N > 0x7fffffff)) return BL_ERR_SHAPE;
  s = check_grid(pl);
  if (s != BL_OK) return s;
  int dev = 0, sms = 0;
  s = current_device(&dev, &sms);
  if (s != BL_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (pl.path == plan::kGemv)
    return run_gemv(pl, dev, sms, xm, act, out_i32, packed, gamma, x, xq, scale, out, acc, st);
  if (pl.path == plan::kSkinny)
    return run_skinny(pl, dev, xm, act, out_i32, packed, gamma, x, xq, scale, out, acc, st);
  return forward_tc(pl, dev, xm, act, out_i32, packed, gamma, x, xq, scale, out, acc, ws, ws_bytes, st);
}

// Device address of g_noalloc_scratch on device `dev` (which must be current).
// In host code the array's name only stands for it; the address is looked up
// once per device and kept.
std::mutex g_noalloc_mu;
void *g_noalloc_ptr[kMaxDevices] = {};

bl_status noalloc_scratch(int dev, void **out) {
  if (dev < 0 || dev >= kMaxDevices) return BL_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (g_noalloc_ptr[dev] == nullptr) {
    void *ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr) {
      cudaGetLastError();
      return BL_ERR_CUDA;
    }
    g_noalloc_ptr[dev] = ptr;
  }
  *out = g_noalloc_ptr[dev];
  return BL_OK;
}

}  // namespace

// ====================================================================== C ABI
extern "C" {

int bitlinear_version(void) { return 100; }

const char *bitlinear_status_string(int status) {
  switch (status) {
    case BL_OK: return "ok";
    case BL_ERR_NULL: return "a required pointer is NULL";
    case BL_ERR_SHAPE: return "a size is outside the supported range";
    case BL_ERR_DTYPE: return "unknown dtype code";
    case BL_ERR_ALIGN: return "a pointer is not suitably aligned";
    case BL_ERR_WORKSPACE: return "workspace missing or too small";
    case BL_ERR_CUDA: return "a CUDA call or kernel launch failed";
    case BL_ERR_UNSUPPORTED: return "the current device is not an sm_103 GPU";
    case BL_ERR_DEVICE: return "a kernel gave up a bounded wait";
    default: return "unknown status";
  }
}

bl_status bitlinear_packed_row_bytes(int64_t K, int64_t *bytes) {
  if (bytes == nullptr) return BL_ERR_NULL;
  if (K < 1 || K > kMaxK) return BL_ERR_SHAPE;
  *bytes = plan::row_bytes(K);
  return BL_OK;
}

bl_status bitlinear_packed_bytes(int64_t N, int64_t K, size_t *bytes) {
  if (bytes == nullptr) return BL_ERR_NULL;
  if (N < 1 || N > kMaxDim || K < 1 || K > kMaxK) return BL_ERR_SHAPE;
  *bytes = static_cast<size_t>(N) * static_cast<size_t>(plan::row_bytes(K));
  return BL_OK;
}

bl_status bitlinear_pack_workspace_bytes(int64_t N, int64_t K, size_t *bytes) {
  if (bytes == nullptr) return BL_ERR_NULL;
  if (N < 1 || N > kMaxDim || K < 1 || K > kMaxK) return BL_ERR_SHAPE;
  *bytes = static_cast<size_t>(N) * sizeof(double);
  return BL_OK;
}

// log2 of a power of two, else -1.
static int log2_exact(int64_t v) {
  if (v < 1 || (v & (v - 1)) != 0) return -1;
  int l = 0;
  while ((int64_t(1) << l) < v) ++l;
  return l;
}

// group_rows 0: one per-tensor scale; otherwise one per group of group_rows rows.
static bl_status pack_common(const void *W, int dtype, int64_t N, int64_t K, int64_t group_rows,
                             uint8_t *packed, float *gamma, void *ws, size_t ws_bytes, void *stream) {
  if (W == nullptr || packed == nullptr || gamma == nullptr) return BL_ERR_NULL;
  if (dtype != BL_F32 && dtype != BL_BF16) return BL_ERR_DTYPE;
  if (N < 1 || N > kMaxDim || K < 1 || K > kMaxK) return BL_ERR_SHAPE;
  const int glog2 = group_rows == 0 ? -1 : log2_exact(group_rows);
  if (group_rows != 0 && (glog2 < 0 || N % group_rows != 0)) return BL_ERR_SHAPE;
  if (ws == nullptr || ws_bytes < static_cast<size_t>(N) * sizeof(double)) return BL_ERR_WORKSPACE;
  if (!aligned(packed, 16) || !aligned(ws, 8) || !aligned(gamma, 4)) return BL_ERR_ALIGN;
  int dev = 0;
  bl_status s = current_device(&dev, nullptr);
  if (s != BL_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  double *rowsum = static_cast<double *>(ws);
  const int64_t wpr = plan::row_bytes(K) / 4;
  const unsigned gsum = static_cast<unsigned>((N + 255) / 256);
  const unsigned gcode = static_cast<unsigned>((N * wpr + 255) / 256);
  uint32_t *pw = reinterpret_cast<uint32_t *>(packed);
  if (dtype == BL_F32)
    s = launch(&pack_rowsum_kernel<float>, dim3(gsum), dim3(256), 0, st, false, static_cast<const float *>(W),
               N, K, rowsum);
  else
    s = launch(&pack_rowsum_kernel<__nv_bfloat16>, dim3(gsum), dim3(256), 0, st, false,
               static_cast<const __nv_bfloat16 *>(W), N, K, rowsum);
  if (s != BL_OK) return s;
  if (group_rows == 0) {
    s = launch(&pack_gamma_kernel, dim3(1), dim3(32), 0, st, false, static_cast<const double *>(rowsum), N, K,
               gamma);
  } else {
    const int64_t groups = N / group_rows;
    s = launch(&pack_gamma_groups_kernel, dim3(static_cast<unsigned>((groups + 127) / 128)), dim3(128), 0, st,
               false, static_cast<const double *>(rowsum), groups, group_rows, K, gamma);
  }
  if (s != BL_OK) return s;
  if (dtype == BL_F32)
    return launch(&pack_codes_kernel<float>, dim3(gcode), dim3(256), 0, st, false, static_cast<const float *>(W),
                  N, K, wpr, static_cast<const float *>(gamma), glog2, pw);
  return launch(&pack_codes_kernel<__nv_bfloat16>, dim3(gcode), dim3(256), 0, st, false,
                static_cast<const __nv_bfloat16 *>(W), N, K, wpr, static_cast<const float *>(gamma), glog2, pw);
}

bl_status bitlinear_pack_weights(const void *W, int dtype, int64_t N, int64_t K, uint8_t *packed,
                                 float *gamma, void *ws, size_t ws_bytes, void *stream) {
  return pack_common(W, dtype, N, K, 0, packed, gamma, ws, ws_bytes, stream);
}

bl_status bitlinear_pack_weights_grouped(const void *W, int dtype, int64_t N, int64_t K, int64_t group_rows,
                                         uint8_t *packed, float *gamma, void *ws, size_t ws_bytes,
                                         void *stream) {
  if (group_rows < 1) return BL_ERR_SHAPE;
  return pack_common(W, dtype, N, K, group_rows, packed, gamma, ws, ws_bytes, stream);
}

static bl_status quant_common(const void *x, int dtype, const float *g, float eps, bool norm, int64_t M,
                              int64_t K, int8_t *xq, float *scale, void *stream, int act = kActNone) {
  if (x == nullptr || xq == nullptr || scale == nullptr) return BL_ERR_NULL;
  if (dtype != BL_F32 && dtype != BL_BF16) return BL_ERR_DTYPE;
  if (M < 1 || M > kMaxDim || K < 1 || K > kMaxK) return BL_ERR_SHAPE;
  if (norm && !(eps >= 0.0f)) return BL_ERR_SHAPE;
  int dev = 0;
  bl_status s = current_device(&dev, nullptr);
  if (s != BL_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const bool ov = g_overlap.load() != 0;
  const dim3 grid(static_cast<unsigned>(M));
  __nv_bfloat16 *nob = nullptr;
  int32_t *noz = nullptr;
  unsigned *noc = nullptr;
  if (dtype == BL_F32) {
    const float *xx = static_cast<const float *>(x);
    if (norm)
      return launch(&quant_act_kernel<float, false, true>, grid, dim3(256), 0, st, ov, xx, K, K, g, eps, xq,
                    nob, scale, noz, int64_t(0), noc, 0, kActNone);
    return launch(&quant_act_kernel<float, false, false>, grid, dim3(256), 0, st, ov, xx, K, K, g, eps, xq,
                  nob, scale, noz, int64_t(0), noc, 0, act);
  }
  const __nv_bfloat16 *xx = static_cast<const __nv_bfloat16 *>(x);
  if (norm)
    return launch(&quant_act_kernel<__nv_bfloat16, false, true>, grid, dim3(256), 0, st, ov, xx, K, K, g,
                  eps, xq, nob, scale, noz, int64_t(0), noc, 0, kActNone);
  return launch(&quant_act_kernel<__nv_bfloat16, false, false>, grid, dim3(256), 0, st, ov, xx, K, K, g,
                eps, xq, nob, scale, noz, int64_t(0), noc, 0, act);
}

bl_status bitlinear_quant_act(const void *x, int dtype, int64_t M, int64_t K, int8_t *xq, float *scale,
                              void *stream) {
  return quant_common(x, dtype, nullptr, 0.0f, false, M, K, xq, scale, stream);
}

bl_status bitlinear_rmsnorm_quant_act(const void *x, int dtype, const float *g, float eps, int64_t M,
                                      int64_t K, int8_t *xq, float *scale, void *stream) {
  return quant_common(x, dtype, g, eps, true, M, K, xq, scale, stream);
}

bl_status bitlinear_workspace_bytes(int64_t M, int64_t N, int64_t K, size_t *bytes) {
  if (bytes == nullptr) return BL_ERR_NULL;
  bl_status s = check_dims(M, N, K);
  if (s != BL_OK) return s;
  const plan::Plan pl = plan::make(M, N, K);
  s = check_grid(pl);
  if (s != BL_OK) return s;
  *bytes = pl.ws_bytes;
  return BL_OK;
}

bl_status bitlinear_forward(const uint8_t *packed, const float *gamma, int64_t N, int64_t K, const void *x,
                            int dtype, int64_t M, float *y, void *ws, size_t ws_bytes, void *stream) {
  if (dtype != BL_F32 && dtype != BL_BF16) return BL_ERR_DTYPE;
  const int xm = dtype == BL_F32 ? gemv::kXF32 : gemv::kXBF16;
  if (y == nullptr) return BL_ERR_NULL;
  return forward_common(packed, gamma, N, K, xm, kActNone, x, nullptr, nullptr, M, out_f32(y), nullptr, ws,
                        ws_bytes, stream);
}

bl_status bitlinear_forward_q(const uint8_t *packed, const float *gamma, int64_t N, int64_t K,
                              const int8_t *xq, const float *scale, int64_t M, float *y, void *ws,
                              size_t ws_bytes, void *stream) {
  if (y == nullptr) return BL_ERR_NULL;
  return forward_common(packed, gamma, N, K, gemv::kXInt8, kActNone, nullptr, xq, scale, M, out_f32(y), nullptr,
                        ws, ws_bytes,
                        stream);
}

bl_status bitlinear_matmul_i32(const uint8_t *packed, int64_t N, int64_t K, const int8_t *xq, int64_t M,
                               int32_t *acc, void *ws, size_t ws_bytes, void *stream) {
  if (acc == nullptr) return BL_ERR_NULL;
  return forward_common(packed, nullptr, N, K, gemv::kXInt8, kActNone, nullptr, xq, nullptr, M,
                        OutSpec{nullptr, nullptr, 0}, acc, ws,
                        ws_bytes, stream);
}

bl_status bitlinear_forward_ex(const uint8_t *packed, const float *gamma, int64_t N, int64_t K, const void *x,
                               int x_dtype, int64_t M, int act, void *y, int y_dtype, const void *residual,
                               void *ws, size_t ws_bytes, void *stream) {
  if (x_dtype != BL_F32 && x_dtype != BL_BF16) return BL_ERR_DTYPE;
  if (y_dtype != BL_F32 && y_dtype != BL_BF16) return BL_ERR_DTYPE;
  if (act != BL_ACT_NONE && act != BL_ACT_RELU2) return BL_ERR_SHAPE;
  if (y == nullptr) return BL_ERR_NULL;
  const int xm = x_dtype == BL_F32 ? gemv::kXF32 : gemv::kXBF16;
  const OutSpec out{y, residual, y_dtype == BL_BF16 ? 1 : 0};
  return forward_common(packed, gamma, N, K, xm, act == BL_ACT_RELU2 ? kActRelu2 : kActNone, x, nullptr, nullptr,
                        M, out, nullptr, ws, ws_bytes, stream);
}
bl_status bitlinear_forward_grouped(const uint8_t *packed, const float *gamma, int64_t group_rows, int64_t N,
                                    int64_t K, const void *x, int x_dtype, int64_t M, int act, void *y,
                                    int y_dtype, const void *residual, void *ws, size_t ws_bytes, void *stream) {
  if (x_dtype != BL_F32 && x_dtype != BL_BF16) return BL_ERR_DTYPE;
  if (y_dtype != BL_F32 && y_dtype != BL_BF16) return BL_ERR_DTYPE;
  if (act != BL_ACT_NONE && act != BL_ACT_RELU2) return BL_ERR_SHAPE;
  if (y == nullptr || gamma == nullptr) return BL_ERR_NULL;
  const int glog2 = log2_exact(group_rows);
  if (glog2 < 0 || N < 1 || N % group_rows != 0) return BL_ERR_SHAPE;
  if (!aligned(gamma, 4)) return BL_ERR_ALIGN;
  const int xm = x_dtype == BL_F32 ? gemv::kXF32 : gemv::kXBF16;
  OutSpec out{y, residual, y_dtype == BL_BF16 ? 1 : 0};
  out.gvec = gamma;
  out.glog2 = glog2;
  return forward_common(packed, gamma, N, K, xm, act == BL_ACT_RELU2 ? kActRelu2 : kActNone, x, nullptr, nullptr,
                        M, out, nullptr, ws, ws_bytes, stream);
}
bl_status bitlinear_forward_relu2(const uint8_t *packed, const float *gamma, int64_t N, int64_t K,
                                  const void *x, int dtype, int64_t M, float *y, void *ws, size_t ws_bytes,
                                  void *stream) {
  if (dtype != BL_F32 && dtype != BL_BF16) return BL_ERR_DTYPE;
  const int xm = dtype == BL_F32 ? gemv::kXF32 : gemv::kXBF16;
  if (y == nullptr) return BL_ERR_NULL;
  return forward_common(packed, gamma, N, K, xm, kActRelu2, x, nullptr, nullptr, M, out_f32(y), nullptr, ws,
                        ws_bytes, stream);
}
bl_status bitlinear_relu2_quant_act(const void *x, int dtype, int64_t M, int64_t K, int8_t *xq, float *scale,
                                    void *stream) {
  return quant_common(x, dtype, nullptr, 0.0f, false, M, K, xq, scale, stream, kActRelu2);
}
// Packed rows [N, rb] bytes as 8-byte elements, read in boxes of `pieces`
// 16-byte pieces (2 elements each) x box_rows rows, unswizzled (the decode
// chain's one-lane-per-row layout: an odd piece count per row keeps the
// lanes' reads on different bank groups), zeros outside the rows.
bool make_map_rows(CUtensorMap *m, const void *ptr, int64_t N, int64_t rb, int pieces, int box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(rb / 8), static_cast<cuuint64_t>(N)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(rb)};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(pieces * (chain::kPiece / 8)), static_cast<cuuint32_t>(box_rows)};
  cuuint32_t es[2] = {1u, 1u};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT64, 2, const_cast<void *>(ptr), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Plan of a decode chain (host): each call's 32-row groups, dealt to the
// blocks round-robin from where the previous call's deal ended (group j of
// call i goes to block (g0_i + j) mod grid), and its tensor map; where its input comes from (quantised ahead into a record, an
// earlier call's output words, or memory after a grid barrier); the workspace
// layout (control words, call table, records, output words).
// Dependencies are read off the calls' buffers:
//   * x written by no earlier call (and no wait_prev): quantised before the
//     chain starts, into a record;
//   * x inside an earlier call's y (fp32, the latest earlier writer of any of
//     x's bytes): read from that call's output words (it writes them);
//   * any other input byte (x, packed, gamma) written by an earlier call, an
//     output byte written or read (from memory) by an earlier call, or
//     wait_prev: a grid barrier before the call.
// A call's output may not overlap its own inputs.  p and t may be null
// (size only).
static int toks(const bl_chain_call &c) { return c.M < 1 ? 1 : c.M; }

static bl_status chain_plan(const bl_chain_call *calls, int n, int grid, chain::Params *p, chain::TableCopy *t,
                            size_t *ws_need, void *ws) {
  if (calls == nullptr) return BL_ERR_NULL;
  if (n < 1 || n > chain::kMaxCalls) return BL_ERR_SHAPE;
  struct Rng {
    uintptr_t lo, hi;
  };
  auto ovl = [](const Rng &a, const Rng &b) { return a.lo < b.hi && b.lo < a.hi; };
  std::vector<Rng> xr(n), yr(n), pr(n), gr(n);
  for (int i = 0; i < n; ++i) {
    const bl_chain_call &c = calls[i];
    if (c.packed == nullptr || c.gamma == nullptr || c.x == nullptr || c.y == nullptr) return BL_ERR_NULL;
    if (c.x_dtype != BL_F32 && c.x_dtype != BL_BF16) return BL_ERR_DTYPE;
    if (c.N < 1 || c.N > chain::kMaxN || c.K < 1 || c.K > chain::kMaxK) return BL_ERR_SHAPE;
    if (c.act != BL_ACT_NONE && c.act != BL_ACT_RELU2) return BL_ERR_SHAPE;
    if (c.M < 0 || c.M > chain::kMaxTok) return BL_ERR_SHAPE;
    if (!aligned(c.packed, 16) || !aligned(c.gamma, 4) || !aligned(c.y, 4)) return BL_ERR_ALIGN;
    const uintptr_t es = c.x_dtype == BL_BF16 ? 2 : 4;
    const uintptr_t m = static_cast<uintptr_t>(toks(c));
    xr[i] = {reinterpret_cast<uintptr_t>(c.x), reinterpret_cast<uintptr_t>(c.x) + m * static_cast<uintptr_t>(c.K) * es};
    yr[i] = {reinterpret_cast<uintptr_t>(c.y), reinterpret_cast<uintptr_t>(c.y) + m * static_cast<uintptr_t>(c.N) * 4};
    pr[i] = {reinterpret_cast<uintptr_t>(c.packed),
             reinterpret_cast<uintptr_t>(c.packed) + static_cast<uintptr_t>(c.N * plan::row_bytes(c.K))};
    gr[i] = {reinterpret_cast<uintptr_t>(c.gamma), reinterpret_cast<uintptr_t>(c.gamma) + 4};
    if (ovl(yr[i], xr[i]) || ovl(yr[i], pr[i]) || ovl(yr[i], gr[i])) return BL_ERR_SHAPE;
  }
  std::vector<int> src(n, -1);
  std::vector<char> produces(n, 0), barrier(n, 0), early(n, 0);
  for (int c = 0; c < n; ++c) {
    bool bar = c > 0 && calls[c].wait_prev != 0;
    int j = -1;
    for (int i = c - 1; i >= 0; --i)
      if (ovl(yr[i], xr[c])) {
        j = i;
        break;
      }
    if (j >= 0) {
      if (calls[c].x_dtype == BL_F32 && toks(calls[c]) == 1 && toks(calls[j]) == 1 && xr[c].lo >= yr[j].lo &&
          xr[c].hi <= yr[j].hi && (xr[c].lo - yr[j].lo) % 4 == 0) {
        src[c] = j;
        produces[j] = 1;
      } else {
        bar = true;
      }
    }
    for (int i = 0; i < c && !bar; ++i) {
      if (ovl(yr[i], pr[c]) || ovl(yr[i], gr[c]) || ovl(yr[c], yr[i]) || ovl(yr[c], pr[i]) ||
          ovl(yr[c], gr[i]) || (src[i] < 0 && ovl(yr[c], xr[i])))
        bar = true;
    }
    barrier[c] = bar ? 1 : 0;
    early[c] = (j < 0 && !bar) ? 1 : 0;  // no earlier call writes x: quantised before the chain
    if (toks(calls[c]) > 1 && !early[c]) return BL_ERR_SHAPE;  // many tokens: only a quantised-ahead input
  }
  size_t off = plan::align256(chain::kTableOffset + static_cast<size_t>(n) * sizeof(chain::Call));
  std::vector<size_t> rec_off(n, 0), mb_off(n, 0);
  for (int i = 0; i < n; ++i)
    if (early[i]) {
      rec_off[i] = off;
      off = plan::align256(off + static_cast<size_t>(chain::record_bytes(static_cast<int>(plan::row_bytes(calls[i].K)),
                                                                         toks(calls[i]))));
    }
  for (int i = 0; i < n; ++i)
    if (produces[i]) {
      mb_off[i] = off;
      off = plan::align256(off + static_cast<size_t>(calls[i].N) * 8);
    }
  *ws_need = off;
  if (p == nullptr) return BL_OK;
  uint8_t *wsb = static_cast<uint8_t *>(ws);
  p->n = n;
  p->ctl = static_cast<unsigned *>(ws);
  p->table = reinterpret_cast<const chain::Call *>(wsb + chain::kTableOffset);
  t->n = n;
  t->dst = reinterpret_cast<chain::Call *>(wsb + chain::kTableOffset);
  int64_t deal = 0;  // the block that takes the next call's group 0
  for (int i = 0; i < n; ++i) {
    const bl_chain_call &c = calls[i];
    chain::Call &d = t->calls[i];
    const int64_t rb = plan::row_bytes(c.K);
    const int64_t ng = (c.N + chain::kGroupRows - 1) / chain::kGroupRows;
    const int P = chain::slab_pieces(static_cast<int>(rb), toks(c));
    if (!make_map_rows(&p->maps[i], c.packed, c.N, rb, P, chain::kGroupRows)) return BL_ERR_CUDA;
    d.gamma = c.gamma;
    d.x = c.x;
    d.y = c.y;
    d.N = static_cast<int>(c.N);
    d.K = static_cast<int>(c.K);
    d.rb = static_cast<int>(rb);
    d.g0 = static_cast<int>(deal);
    d.ng = static_cast<int>(ng);
    deal = (deal + ng) % grid;
    const int flags = (c.x_dtype == BL_BF16 ? chain::kFlagBf16 : 0) | (c.act == BL_ACT_RELU2 ? chain::kFlagRelu2 : 0);
    d.flags = flags | (barrier[i] ? chain::kFlagBarrier : 0);
    d.src = src[i];
    d.M = toks(c);
    d.P = P;
    d.ns = chain::slabs_of(static_cast<int>(rb), toks(c));
    d.rec = early[i] ? wsb + rec_off[i] : nullptr;
    d.mb_out = produces[i] ? reinterpret_cast<uint64_t *>(wsb + mb_off[i]) : nullptr;
    d.mb_in = nullptr;
  }
  for (int i = 0; i < n; ++i)
    if (src[i] >= 0)
      t->calls[i].mb_in = t->calls[src[i]].mb_out + (xr[i].lo - yr[src[i]].lo) / 4;
  return BL_OK;
}

bl_status bitlinear_chain_workspace_bytes(const bl_chain_call *calls, int n, size_t *bytes) {
  if (bytes == nullptr) return BL_ERR_NULL;
  size_t need = 0;
  bl_status s = chain_plan(calls, n, 1, nullptr, nullptr, &need, nullptr);
  if (s != BL_OK) return s;
  *bytes = need;
  return BL_OK;
}

bl_status bitlinear_forward_chain(const bl_chain_call *calls, int n, void *ws, size_t ws_bytes,
                                  void *stream) {
  if (calls == nullptr || ws == nullptr) return BL_ERR_NULL;
  if (!aligned(ws, 256)) return BL_ERR_ALIGN;
  size_t need = 0;
  bl_status s = chain_plan(calls, n, 1, nullptr, nullptr, &need, nullptr);
  if (s != BL_OK) return s;
  if (ws_bytes < need) return BL_ERR_WORKSPACE;
  int dev = 0, sms = 0;
  s = current_device(&dev, &sms);
  if (s != BL_OK) return s;
  // about 30 KB of tensor maps and 21 KB of call table: kept off the stack
  // (each launch copies its parameters)
  static chain::Params p;
  static chain::TableCopy tc;
  static std::mutex p_mu;
  std::lock_guard<std::mutex> lk(p_mu);
  s = chain_plan(calls, n, sms, &p, &tc, &need, ws);
  if (s != BL_OK) return s;
  bool many = false;
  for (int i = 0; i < n; ++i) many = many || toks(calls[i]) > 1;
  bool dep = false;  // a call whose input an earlier call writes (quantised in the block)
  for (int i = 0; i < n; ++i) dep = dep || tc.calls[i].rec == nullptr;
  void (*kern)(chain::Params) =
      many ? (dep ? &chain::chain_kernel<true, true> : &chain::chain_kernel<true, false>)
           : (dep ? &chain::chain_kernel<false, true> : &chain::chain_kernel<false, false>);
  const int smem = chain::smem_bytes(many, dep);
  s = ensure_smem(dev, reinterpret_cast<const void *>(kern), smem);
  if (s != BL_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // the call table into the workspace (its parameters are kept by value)
  // and the inputs no earlier call writes quantised into their records, one
  // launch: block (i, m) takes token m of call i
  int mt = 1;
  for (int i = 0; i < n; ++i)
    if (tc.calls[i].rec != nullptr && tc.calls[i].M > mt) mt = tc.calls[i].M;
  s = launch(&chain::chain_setup_kernel, dim3(static_cast<unsigned>(n), static_cast<unsigned>(mt)),
             dim3(chain::kQThreads), 0, st, false, tc);
  if (s != BL_OK) return s;
  // every block may wait for the others: all must be resident (one per SM)
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(sms));
  cfg.blockDim = dim3(chain::kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  // and it may start while the set-up kernel runs: it waits for it
  // (griddepcontrol) after initialising its barriers
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  if (cudaLaunchKernelEx(&cfg, kern, p) != cudaSuccess) {
    cudaGetLastError();  // not taken with the overlap: launch in plain stream order
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, kern, p) != cudaSuccess) return launch_failed("chain launch");
  }
  return BL_OK;
}
bl_status bitlinear_forward_noalloc(const uint8_t *packed, const float *gamma, int64_t N, int64_t K,
                                    const void *x, int dtype, int64_t M, float *y, void *stream) {
  if (dtype != BL_F32 && dtype != BL_BF16) return BL_ERR_DTYPE;
  if (packed == nullptr || gamma == nullptr || x == nullptr || y == nullptr) return BL_ERR_NULL;
  bl_status s = check_dims(M, N, K);
  if (s != BL_OK) return s;
  const plan::Plan pl = plan::make(M, N, K);
  s = check_grid(pl);
  if (s != BL_OK) return s;
  const size_t need = pl.ws_bytes;
  if (need > kNoAllocScratchBytes) return BL_ERR_WORKSPACE;
  void *ws = nullptr;
  if (need > 0) {
    int dev = 0;
    s = current_device(&dev, nullptr);
    if (s != BL_OK) return s;
    s = noalloc_scratch(dev, &ws);
    if (s != BL_OK) return s;
  }
  return bitlinear_forward(packed, gamma, N, K, x, dtype, M, y, ws, need > 0 ? kNoAllocScratchBytes : 0,
                           stream);
}

void bitlinear_set_launch_overlap(int mode) { g_overlap.store(mode < 0 ? 0 : (mode > 2 ? 2 : mode)); }

int bitlinear_get_launch_overlap(void) { return g_overlap.load(); }

bl_status bitlinear_device_error(unsigned int *flags, int clear) {
  if (flags == nullptr) return BL_ERR_NULL;
  unsigned v = 0;
  if (cudaMemcpyFromSymbol(&v, bl::g_dev_error, sizeof(v)) != cudaSuccess) {
    cudaGetLastError();
    return BL_ERR_CUDA;
  }
  if (clear && v != 0) {
    const unsigned z = 0;
    if (cudaMemcpyToSymbol(bl::g_dev_error, &z, sizeof(z)) != cudaSuccess) {
      cudaGetLastError();
      return BL_ERR_CUDA;
    }
  }
  *flags = v;
  return v ? BL_ERR_DEVICE : BL_OK;
}

}  // extern "C"
