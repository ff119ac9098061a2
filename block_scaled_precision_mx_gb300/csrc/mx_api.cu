// mx_api.cu -- the C ABI declared in include/mx.h: host-side validation, TMA descriptor
// encoding and kernel launches.  This is the only translation unit of libmxgb.so; the kernels
// are included from the .cuh files so that the device error word needs no separate linking.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "../../include/mx.h"
#include "mx_device.cuh"
#include "mx_gemm.cuh"
#include "mx_gemm2.cuh"
#include "mx_quantize.cuh"

using namespace mxgb;

namespace {

constexpr int kAbiVersion = 1;

inline bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

inline cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }

mx_status launch_status() {
  const cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? MX_OK : MX_ERR_CUDA;
}

// The quantizers and small helper kernels are launched with programmatic stream serialization:
// one may be scheduled while the previous kernel on the stream finishes (each allows it at its
// start) and waits for that kernel to complete before it reads memory, so dependent calls stay
// ordered and the launch latency overlaps the previous kernel's last wave.  The GEMMs take no
// part: they are launched the ordinary way and do not let the next kernel start early.  Their
// persistent CTAs take tiles in a fixed order; early-started CTAs on the SMs a previous kernel
// left first, or a next kernel's CTAs waiting on SMs the GEMM left first, made a full step 3-5%
// slower in both cases.
template <typename Kern, typename... Args>
cudaError_t pdl_launch(Kern kern, dim3 grid, dim3 block, size_t smem, cudaStream_t st, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute a[1];
  a[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  a[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = a;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

// ---------------------------------------------------------------- driver entry point
PFN_cuTensorMapEncodeTiled_v12000 get_encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 2-D tensor maps, remembered: a map depends only on the arguments of its encoding (address,
// shape, stride, box, element type, swizzle, L2 promotion), so repeated calls on the same buffers
// (a training step, a benchmark loop) copy a stored map instead of encoding it again.  A small
// direct-mapped table under a mutex; a slot holds the last map whose key hashed there.
struct TmapKey {
  const void* base;
  uint64_t dim0, dim1, stride;
  uint32_t box0, box1;
  int dtype, swizzle, promo;
  bool operator==(const TmapKey& o) const {
    return base == o.base && dim0 == o.dim0 && dim1 == o.dim1 && stride == o.stride && box0 == o.box0 &&
           box1 == o.box1 && dtype == o.dtype && swizzle == o.swizzle && promo == o.promo;
  }
};
struct TmapSlot {
  TmapKey key;
  CUtensorMap map;
  bool valid;
};
constexpr int kTmapSlots = 256;
TmapSlot g_tmaps[kTmapSlots];
std::mutex g_tmap_mu;

bool encode_2d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base, uint64_t dim0, uint64_t dim1,
               uint64_t stride, uint32_t box0, uint32_t box1, CUtensorMapSwizzle swizzle,
               CUtensorMapL2promotion promo) {
  const TmapKey key{base, dim0, dim1, stride, box0, box1, static_cast<int>(dtype), static_cast<int>(swizzle),
                    static_cast<int>(promo)};
  uint64_t h = reinterpret_cast<uintptr_t>(base) >> 8;
  h ^= dim0 * 0x9E3779B97F4A7C15ull ^ dim1 * 0xC2B2AE3D27D4EB4Full ^ (static_cast<uint64_t>(box1) << 20) ^
       static_cast<uint64_t>(swizzle) * 131 ^ static_cast<uint64_t>(dtype) * 977;
  TmapSlot& slot = g_tmaps[(h ^ (h >> 29)) % kTmapSlots];
  {
    std::lock_guard<std::mutex> lock(g_tmap_mu);
    if (slot.valid && slot.key == key) {
      *map = slot.map;
      return true;
    }
  }
  auto fn = get_encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {dim0, dim1};
  cuuint64_t strides[1] = {stride};
  cuuint32_t box[2] = {box0, box1};
  cuuint32_t estr[2] = {1u, 1u};
  if (fn(map, dtype, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
         promo, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return false;
  std::lock_guard<std::mutex> lock(g_tmap_mu);
  slot.key = key;
  slot.map = *map;
  slot.valid = true;
  return true;
}

// 2-D byte tensor [rows][row_bytes], box 128 bytes x box_rows, 128-byte swizzle (swizzle=false:
// unswizzled, used for scale chunks read as 128-byte rows).
bool make_tmap(CUtensorMap* map, const void* base, int64_t rows, int64_t row_bytes, int box_rows,
               bool swizzle = true) {
  return encode_2d(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, base, static_cast<uint64_t>(row_bytes),
                   static_cast<uint64_t>(rows), static_cast<uint64_t>(row_bytes), 128u,
                   static_cast<uint32_t>(box_rows), swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
}

// ---------------------------------------------------------------- device properties
// Per-device caches, filled on first use; atomics so that host threads calling concurrently
// read and write them without a data race (they all compute the same values).
struct DevInfo {
  std::atomic<int> sms{0};
};
DevInfo g_dev[64];
std::atomic<int> g_last_sms{0};

int device_sms() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  int n = g_dev[dev].sms.load(std::memory_order_relaxed);
  if (n == 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    g_dev[dev].sms.store(n, std::memory_order_relaxed);
  }
  g_last_sms.store(n, std::memory_order_relaxed);
  return n;
}

// ---------------------------------------------------------------- GEMM launch
template <int KIND, int BN, bool OUT_BF16>
mx_status launch_gemm(const void* qa, const void* qb, int64_t kbytes, const GemmArgs& args, cudaStream_t st) {
  using Cfg = GemmCfg<KIND, BN>;
  auto kern = bs_gemm_kernel<KIND, BN, OUT_BF16>;
  static std::atomic<bool> attr_set[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return MX_ERR_CUDA;
  if (!attr_set[dev].load(std::memory_order_relaxed)) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM_BYTES) != cudaSuccess)
      return MX_ERR_CUDA;
    attr_set[dev].store(true, std::memory_order_relaxed);
  }
  CUtensorMap ta, tb;
  if (!make_tmap(&ta, qa, args.M, kbytes, Cfg::BM)) return MX_ERR_CUDA;
  if (!make_tmap(&tb, qb, args.N, kbytes, BN)) return MX_ERR_CUDA;
  const int sms = device_sms();
  if (sms <= 0) return MX_ERR_CUDA;
  const int tiles = (args.M / Cfg::BM) * (args.N / BN);
  const int grid = tiles < sms ? tiles : sms;
  kern<<<grid, Cfg::THREADS, Cfg::SMEM_BYTES, st>>>(ta, tb, args);  // not a dependent launch (see above)
  return launch_status();
}

// Output tensor map: [M][ldc] elements, 32 x 32 boxes, swizzle matching the epilogues' staging
// layout (64-byte rows for bf16, 128-byte rows for FP32).
bool make_out_tmap(CUtensorMap* map, void* out, int64_t M, int64_t N, int64_t ldc, bool bf16) {
  const uint64_t es = bf16 ? 2 : 4;
  return encode_2d(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, out,
                   static_cast<uint64_t>(N), static_cast<uint64_t>(M), static_cast<uint64_t>(ldc) * es, 32u, 32u,
                   bf16 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE);
}

// Launch a CTA-pair kernel: clusters of two CTAs, as many clusters as fit on the device at once
// (each persistent over its share of `tiles`).  `max_clusters` caches the occupancy per device
// for this kernel.
template <typename... KArgs, typename... Args>
mx_status launch_pairs(void (*kern)(KArgs...), int threads, int smem_bytes, int tiles,
                       std::atomic<int> (&max_clusters)[64],
                       cudaStream_t st, Args... args) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return MX_ERR_CUDA;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(static_cast<unsigned>(threads));
  cfg.dynamicSmemBytes = static_cast<size_t>(smem_bytes);
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = max_clusters[dev].load(std::memory_order_relaxed);
  if (n == 0) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes) != cudaSuccess)
      return MX_ERR_CUDA;
    const int sms = device_sms();
    cfg.gridDim = dim3(static_cast<unsigned>(sms - (sms & 1)));
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess || n <= 0) return MX_ERR_CUDA;
    max_clusters[dev].store(n, std::memory_order_relaxed);
  }
  const int clusters = tiles < n ? tiles : n;
  cfg.gridDim = dim3(static_cast<unsigned>(2 * clusters));
  if (cudaLaunchKernelEx(&cfg, kern, args...) != cudaSuccess) return MX_ERR_CUDA;
  return launch_status();
}

// Block-scaled CTA-pair kernel, 256 x 256 output tiles.
template <int KIND, bool OUT_BF16, bool GROUPED = false, int MXOUT = -1>
mx_status launch_gemm2(const void* qa, const void* qb, int64_t kbytes, const GemmArgs& args, cudaStream_t st,
                       int64_t b_rows = 0) {
  using Cfg = Gemm2Cfg<KIND, OUT_BF16 || (MXOUT >= 0), GROUPED>;
  static std::atomic<int> max_clusters[64];
  const int64_t kc = (KIND == kNvf4) ? args.K / 64 : args.K / 128;  // 512-byte scale chunks per 128 rows
  const int chunk_rows = Cfg::SF_CHUNK / 128;
  CUtensorMap ta, tb, tsa, tsb, tout;
  if (!make_tmap(&ta, qa, args.M, kbytes, Cfg::ROWS)) return MX_ERR_CUDA;
  const int64_t brows = GROUPED ? b_rows : args.N;  // grouped: the groups' B blocks stacked
  if (!make_tmap(&tb, qb, brows, kbytes, Cfg::ROWS)) return MX_ERR_CUDA;
  if (!make_tmap(&tsa, args.sfa, (args.M / 128) * kc * 4, 128, chunk_rows, false)) return MX_ERR_CUDA;
  if (!make_tmap(&tsb, args.sfb, (brows / 128) * kc * 4, 128, chunk_rows, false)) return MX_ERR_CUDA;
  // (MX output: the epilogue stores codes itself; the map describes a code buffer as FP32 words
  // and is never used)
  const bool ok_out =
      MXOUT < 0 ? make_out_tmap(&tout, args.out, args.M, args.N, args.ldc, OUT_BF16)
      : args.q_out ? make_out_tmap(&tout, args.q_out, args.M, args.N / 4, args.ldc / 4, false)
                   : make_out_tmap(&tout, args.q_col, args.N, args.M / 4, args.ldq_col / 4, false);
  if (!ok_out) return MX_ERR_CUDA;
  // grouped: the tile count is known on the device only; every co-resident cluster runs
  const int tiles = GROUPED ? 0x7FFFFFFF : (args.M / Cfg::BM) * (args.N / Cfg::BN);
  return launch_pairs(bs_gemm2_kernel<KIND, OUT_BF16, GROUPED, MXOUT>, Cfg::THREADS, Cfg::SMEM_BYTES, tiles,
                      max_clusters, st, ta, tb, tsa, tsb, tout, args);
}

// DeepSeek CTA-pair kernel, 256 x 256 output tiles.
template <bool OUT_BF16, bool GROUPED = false>
mx_status launch_ds_gemm2(const void* qa, const void* qb, const GemmArgs& args, cudaStream_t st, int64_t b_rows = 0) {
  using Cfg = Ds2Cfg<OUT_BF16, GROUPED>;
  static std::atomic<int> max_clusters[64];
  CUtensorMap ta, tb, tout;
  if (!make_tmap(&ta, qa, args.M, args.K, Cfg::ROWS)) return MX_ERR_CUDA;
  if (!make_tmap(&tb, qb, GROUPED ? b_rows : args.N, args.K, Cfg::ROWS)) return MX_ERR_CUDA;
  if (!make_out_tmap(&tout, args.out, args.M, args.N, args.ldc, OUT_BF16)) return MX_ERR_CUDA;
  // grouped: the tile count is known on the device only; every co-resident cluster runs
  const int tiles = GROUPED ? 0x7FFFFFFF : (args.M / Cfg::BM) * (args.N / Cfg::BN);
  return launch_pairs(ds_gemm2_kernel<OUT_BF16, GROUPED>, Cfg::THREADS, Cfg::SMEM_BYTES, tiles, max_clusters, st,
                      ta, tb, tout, args);
}

// MX quantize launch: nf = 1 (format f0) or 2 (E4M3 and E5M2 from one read).
// Quantizer grids are 2-D, x = row tiles (< 2^31), y = column tiles (at most 65535), so that no
// thread divides 64-bit integers to find its tile.
bool quant_grid(int64_t row_tiles, int64_t col_tiles, dim3* g) {
  if (row_tiles <= 0 || col_tiles <= 0 || row_tiles > 0x7FFFFFFFll || col_tiles > 65535) return false;
  *g = dim3(static_cast<unsigned>(row_tiles), static_cast<unsigned>(col_tiles));
  return true;
}

mx_status launch_mx_quantize(const uint16_t* x, int64_t rows, int64_t cols, int f0, int nf, bool row, bool col,
                             const MxOut& o, cudaStream_t st, bool b2d = false) {
  dim3 grid;
  if (!quant_grid(rows / 128, cols / 128, &grid)) return MX_ERR_INVALID_ARG;
#define MXQ(F, N, R, C) pdl_launch(mx_quantize_kernel<F, N, R, C>, grid, 256, 0, st, x, rows, cols, o)
#define MXQ2D(F, R, C) pdl_launch(mx_quantize_kernel<F, 1, R, C, true>, grid, 256, 0, st, x, rows, cols, o)
  if (b2d) {  // 2-D 32x32 blocks, MXFP8 only
    if (f0 == 0) {
      if (row && col) MXQ2D(0, true, true);
      else if (row) MXQ2D(0, true, false);
      else MXQ2D(0, false, true);
    } else {
      if (row && col) MXQ2D(1, true, true);
      else if (row) MXQ2D(1, true, false);
      else MXQ2D(1, false, true);
    }
  } else if (nf == 2) {
    if (row && col) MXQ(0, 2, true, true);
    else if (row) MXQ(0, 2, true, false);
    else MXQ(0, 2, false, true);
  } else if (f0 == 0) {
    if (row && col) MXQ(0, 1, true, true);
    else if (row) MXQ(0, 1, true, false);
    else MXQ(0, 1, false, true);
  } else if (f0 == 2) {
    if (row && col) MXQ(2, 1, true, true);
    else if (row) MXQ(2, 1, true, false);
    else MXQ(2, 1, false, true);
  } else {
    if (row && col) MXQ(1, 1, true, true);
    else if (row) MXQ(1, 1, true, false);
    else MXQ(1, 1, false, true);
  }
#undef MXQ
#undef MXQ2D
  return launch_status();
}

bool gemm_shape_ok(int64_t M, int64_t N, int64_t K, int64_t kmult, int64_t ldc, mx_out od) {
  if (M <= 0 || N <= 0 || K <= 0) return false;
  if (M % 128 || N % 128 || K % kmult) return false;
  if (M > (1ll << 30) || N > (1ll << 30) || K > (1ll << 30)) return false;
  if (ldc < N || ldc % 8) return false;
  if (od != MX_OUT_F32 && od != MX_OUT_BF16) return false;
  return true;
}

}  // namespace

extern "C" {

int mx_abi_version(void) { return kAbiVersion; }

const char* mx_status_string(mx_status s) {
  switch (s) {
    case MX_OK: return "MX_OK";
    case MX_ERR_INVALID_ARG: return "MX_ERR_INVALID_ARG";
    case MX_ERR_UNSUPPORTED: return "MX_ERR_UNSUPPORTED";
    case MX_ERR_CUDA: return "MX_ERR_CUDA";
    case MX_ERR_TIMEOUT: return "MX_ERR_TIMEOUT";
  }
  return "MX_ERR_UNKNOWN";
}

int mx_num_sms(void) { return g_last_sms.load(std::memory_order_relaxed); }

size_t mx_scale_bytes(int64_t rows, int64_t cols, int block, int block_rows, mx_scale_fmt sfmt) {
  if (rows <= 0 || cols <= 0) return 0;
  if (block == 32 && (block_rows == 1 || block_rows == 32) && sfmt == MX_SCALE_E8M0)
    return static_cast<size_t>(rows * (cols / 32));  // 32x32 blocks are stored expanded per 1x32
  if (block == 16 && block_rows == 1 && sfmt == MX_SCALE_UE4M3) return static_cast<size_t>(rows * (cols / 16));
  const bool f32 = sfmt == MX_SCALE_FP32 || sfmt == MX_SCALE_FP32_POW2;
  if (block == 128 && block_rows == 1 && f32) return static_cast<size_t>(4 * rows * (cols / 128));
  if (block == 128 && block_rows == 128 && f32)
    return static_cast<size_t>(4 * (rows / 128) * (cols / 128));
  return 0;
}

mx_status mx_quantize(const void* x, int64_t rows, int64_t cols, int block, int block_rows, mx_elem elem,
                      mx_scale_fmt sfmt, mx_layout layout, void* q_row, void* s_row, void* q_col, void* s_col,
                      void* stream) {
  if (!x || rows <= 0 || cols <= 0 || rows % 128 || cols % 128) return MX_ERR_INVALID_ARG;
  if (rows > (1ll << 31) || cols > (1ll << 31)) return MX_ERR_INVALID_ARG;
  if (elem != MX_E4M3 && elem != MX_E5M2 && elem != MX_E2M1) return MX_ERR_INVALID_ARG;
  if (sfmt != MX_SCALE_E8M0 && sfmt != MX_SCALE_UE4M3 && sfmt != MX_SCALE_FP32 && sfmt != MX_SCALE_FP32_POW2)
    return MX_ERR_INVALID_ARG;
  if (layout != MX_ROWWISE && layout != MX_COLWISE && layout != MX_BOTH) return MX_ERR_INVALID_ARG;
  if (!aligned(x, 16)) return MX_ERR_INVALID_ARG;
  cudaStream_t st = as_stream(stream);
  const bool row = (layout & MX_ROWWISE) != 0, col = (layout & MX_COLWISE) != 0;

  const bool b2d = block_rows == 32;  // 2-D 32x32 blocks (MXFP8 weights)
  if (block == 32 && (block_rows == 1 || (b2d && elem != MX_E2M1)) && sfmt == MX_SCALE_E8M0) {
    // MXFP8 (E4M3, E5M2) or MXFP4 (E2M1); 1x32 blocks, or 32x32 blocks for MXFP8
    if (row && (!q_row || !s_row || !aligned(q_row, 16) || !aligned(s_row, 16))) return MX_ERR_INVALID_ARG;
    if (col && (!q_col || !s_col || !aligned(q_col, 16) || !aligned(s_col, 16))) return MX_ERR_INVALID_ARG;
    const int64_t tiles = (rows / 128) * (cols / 128);
    if (tiles > 0x7FFFFFFFll) return MX_ERR_INVALID_ARG;
    MxOut o{};
    o.q_row[0] = static_cast<uint8_t*>(q_row);
    o.s_row[0] = static_cast<uint8_t*>(s_row);
    o.q_col[0] = static_cast<uint8_t*>(q_col);
    o.s_col[0] = static_cast<uint8_t*>(s_col);
    const int f0 = elem == MX_E4M3 ? 0 : (elem == MX_E5M2 ? 1 : 2);
    return launch_mx_quantize(static_cast<const uint16_t*>(x), rows, cols, f0, 1, row, col, o, st, b2d);
  }
  if (block == 128 && (sfmt == MX_SCALE_FP32 || sfmt == MX_SCALE_FP32_POW2) && elem == MX_E4M3 &&
      layout == MX_ROWWISE && (block_rows == 1 || block_rows == 128)) {
    if (!q_row || !s_row || !aligned(q_row, 16) || !aligned(s_row, 4)) return MX_ERR_INVALID_ARG;
    const uint16_t* xb = static_cast<const uint16_t*>(x);
    auto* qo = static_cast<uint8_t*>(q_row);
    auto* so = static_cast<float*>(s_row);
    const bool pow2 = sfmt == MX_SCALE_FP32_POW2;
    dim3 grid;
    if (block_rows == 1) {
      if (!quant_grid(rows / 64, cols / 128, &grid)) return MX_ERR_INVALID_ARG;
      if (pow2) pdl_launch(ds_quantize_1x128_kernel<true>, grid, 256, 0, st, xb, rows, cols, qo, so);
      else pdl_launch(ds_quantize_1x128_kernel<false>, grid, 256, 0, st, xb, rows, cols, qo, so);
    } else {
      if (!quant_grid(rows / 128, cols / 128, &grid)) return MX_ERR_INVALID_ARG;
      CUtensorMap tmx;  // x as bytes [rows][2 cols], boxes of 128 bytes x 128 rows
      if (!make_tmap(&tmx, x, rows, cols * 2, 128, false)) return MX_ERR_CUDA;
      if (pow2) pdl_launch(ds_quantize_128x128_kernel<true>, grid, 256, 0, st, tmx, rows, cols, qo, so);
      else pdl_launch(ds_quantize_128x128_kernel<false>, grid, 256, 0, st, tmx, rows, cols, qo, so);
    }
    return launch_status();
  }
  return MX_ERR_UNSUPPORTED;
}

mx_status mx_quantize_dual(const void* x, int64_t rows, int64_t cols, mx_layout layout, void* q_row_e4m3,
                           void* s_row_e4m3, void* q_col_e4m3, void* s_col_e4m3, void* q_row_e5m2, void* s_row_e5m2,
                           void* q_col_e5m2, void* s_col_e5m2, void* stream) {
  if (!x || rows <= 0 || cols <= 0 || rows % 128 || cols % 128) return MX_ERR_INVALID_ARG;
  if (rows > (1ll << 31) || cols > (1ll << 31)) return MX_ERR_INVALID_ARG;
  if (layout != MX_ROWWISE && layout != MX_COLWISE && layout != MX_BOTH) return MX_ERR_INVALID_ARG;
  if (!aligned(x, 16)) return MX_ERR_INVALID_ARG;
  const bool row = (layout & MX_ROWWISE) != 0, col = (layout & MX_COLWISE) != 0;
  void* rp[4] = {q_row_e4m3, s_row_e4m3, q_row_e5m2, s_row_e5m2};
  void* cp[4] = {q_col_e4m3, s_col_e4m3, q_col_e5m2, s_col_e5m2};
  for (int i = 0; i < 4; ++i) {
    if (row && (!rp[i] || !aligned(rp[i], 16))) return MX_ERR_INVALID_ARG;
    if (col && (!cp[i] || !aligned(cp[i], 16))) return MX_ERR_INVALID_ARG;
  }
  MxOut o{};
  o.q_row[0] = static_cast<uint8_t*>(q_row_e4m3);
  o.s_row[0] = static_cast<uint8_t*>(s_row_e4m3);
  o.q_col[0] = static_cast<uint8_t*>(q_col_e4m3);
  o.s_col[0] = static_cast<uint8_t*>(s_col_e4m3);
  o.q_row[1] = static_cast<uint8_t*>(q_row_e5m2);
  o.s_row[1] = static_cast<uint8_t*>(s_row_e5m2);
  o.q_col[1] = static_cast<uint8_t*>(q_col_e5m2);
  o.s_col[1] = static_cast<uint8_t*>(s_col_e5m2);
  return launch_mx_quantize(static_cast<const uint16_t*>(x), rows, cols, 0, 2, row, col, o, as_stream(stream));
}

mx_status mx_gemm(const void* qa, const void* sa, mx_elem ea, const void* qb, const void* sb, mx_elem eb, int64_t M,
                  int64_t N, int64_t K, void* out, mx_out out_dtype, int64_t ldc, void* stream) {
  if (!qa || !sa || !qb || !sb || !out) return MX_ERR_INVALID_ARG;
  if (!gemm_shape_ok(M, N, K, 128, ldc, out_dtype)) return MX_ERR_INVALID_ARG;
  if (!aligned(qa, 16) || !aligned(qb, 16) || !aligned(sa, 16) || !aligned(sb, 16) || !aligned(out, 16))
    return MX_ERR_INVALID_ARG;
  const bool fp4 = ea == MX_E2M1 && eb == MX_E2M1;  // MXFP4 x MXFP4
  if (!fp4) {
    if ((ea != MX_E4M3 && ea != MX_E5M2 && ea != MX_E2M1) || (eb != MX_E4M3 && eb != MX_E5M2 && eb != MX_E2M1))
      return MX_ERR_INVALID_ARG;
    if (ea == MX_E2M1 || eb == MX_E2M1) return MX_ERR_UNSUPPORTED;  // FP4 x FP8 mixes are not built
  }
  if (fp4 && K % 256) return MX_ERR_INVALID_ARG;  // 256 FP4 elements of K per stage
  GemmArgs a{};
  a.sfa = static_cast<const uint8_t*>(sa);
  a.sfb = static_cast<const uint8_t*>(sb);
  a.out = out;
  a.ldc = ldc;
  a.M = static_cast<int>(M);
  a.N = static_cast<int>(N);
  a.K = static_cast<int>(K);
  const bool bn256 = (N % 256) == 0;
  cudaStream_t st = as_stream(stream);
  const bool bf = out_dtype == MX_OUT_BF16;
  if (fp4) {  // kind::mxf4nvf4 operand type 1 = E2M1, UE8M0 scales; K / 2 bytes per row
    const int64_t kb = K / 2;
    if (bn256 && (M % 256) == 0) {
      a.idesc = make_idesc_block_scaled(1u, 1u, 256, 256, 1);
      return bf ? launch_gemm2<kMxf4, true>(qa, qb, kb, a, st) : launch_gemm2<kMxf4, false>(qa, qb, kb, a, st);
    }
    a.idesc = make_idesc_block_scaled(1u, 1u, 128, bn256 ? 256 : 128, 1);
    if (bn256)
      return bf ? launch_gemm<kMxf4, 256, true>(qa, qb, kb, a, st)
                : launch_gemm<kMxf4, 256, false>(qa, qb, kb, a, st);
    return bf ? launch_gemm<kMxf4, 128, true>(qa, qb, kb, a, st) : launch_gemm<kMxf4, 128, false>(qa, qb, kb, a, st);
  }
  if (bn256 && (M % 256) == 0) {
    a.idesc = make_idesc_block_scaled(static_cast<uint32_t>(ea), static_cast<uint32_t>(eb), 256, 256, 1);
    return bf ? launch_gemm2<kMxf8, true>(qa, qb, K, a, st) : launch_gemm2<kMxf8, false>(qa, qb, K, a, st);
  }
  a.idesc = make_idesc_block_scaled(static_cast<uint32_t>(ea), static_cast<uint32_t>(eb), 128, bn256 ? 256 : 128, 1);
  if (bn256)
    return bf ? launch_gemm<kMxf8, 256, true>(qa, qb, K, a, st)
              : launch_gemm<kMxf8, 256, false>(qa, qb, K, a, st);
  return bf ? launch_gemm<kMxf8, 128, true>(qa, qb, K, a, st) : launch_gemm<kMxf8, 128, false>(qa, qb, K, a, st);
}

mx_status mx_gemm_mxout_ex(const void* qa, const void* sa, mx_elem ea, const void* qb, const void* sb, mx_elem eb,
                           int64_t M, int64_t N, int64_t K, mx_elem out_elem, mx_layout layout, void* q_row,
                           void* s_row, int64_t ldq_row, void* q_col, void* s_col, int64_t ldq_col, void* stream) {
  if (layout != MX_ROWWISE && layout != MX_COLWISE && layout != MX_BOTH) return MX_ERR_INVALID_ARG;
  const bool row = layout & MX_ROWWISE, col = layout & MX_COLWISE;
  if (!qa || !sa || !qb || !sb) return MX_ERR_INVALID_ARG;
  if (row && (!q_row || !s_row)) return MX_ERR_INVALID_ARG;
  if (col && (!q_col || !s_col)) return MX_ERR_INVALID_ARG;
  if (M <= 0 || N <= 0 || K <= 0 || M % 256 || N % 256 || K % 128) return MX_ERR_INVALID_ARG;
  if (M > (1ll << 30) || N > (1ll << 30) || K > (1ll << 30)) return MX_ERR_INVALID_ARG;
  if (row && (ldq_row < N || ldq_row % 16)) return MX_ERR_INVALID_ARG;
  if (col && (ldq_col < M || ldq_col % 16)) return MX_ERR_INVALID_ARG;
  if (!aligned(qa, 16) || !aligned(qb, 16) || !aligned(sa, 16) || !aligned(sb, 16)) return MX_ERR_INVALID_ARG;
  if (row && (!aligned(q_row, 16) || !aligned(s_row, 16))) return MX_ERR_INVALID_ARG;
  if (col && (!aligned(q_col, 16) || !aligned(s_col, 16))) return MX_ERR_INVALID_ARG;
  if ((ea != MX_E4M3 && ea != MX_E5M2) || (eb != MX_E4M3 && eb != MX_E5M2)) {
    if (ea == MX_E2M1 || eb == MX_E2M1) return MX_ERR_UNSUPPORTED;
    return MX_ERR_INVALID_ARG;
  }
  if (out_elem != MX_E4M3 && out_elem != MX_E5M2) return out_elem == MX_E2M1 ? MX_ERR_UNSUPPORTED : MX_ERR_INVALID_ARG;
  GemmArgs a{};
  a.sfa = static_cast<const uint8_t*>(sa);
  a.sfb = static_cast<const uint8_t*>(sb);
  a.q_out = row ? static_cast<uint8_t*>(q_row) : nullptr;
  a.s_out = row ? static_cast<uint8_t*>(s_row) : nullptr;
  a.ldc = row ? ldq_row : N;
  a.q_col = col ? static_cast<uint8_t*>(q_col) : nullptr;
  a.s_col = col ? static_cast<uint8_t*>(s_col) : nullptr;
  a.ldq_col = ldq_col;
  a.M = static_cast<int>(M);
  a.N = static_cast<int>(N);
  a.K = static_cast<int>(K);
  a.idesc = make_idesc_block_scaled(static_cast<uint32_t>(ea), static_cast<uint32_t>(eb), 256, 256, 1);
  cudaStream_t st = as_stream(stream);
  const bool e4 = out_elem == MX_E4M3;
  if (layout == MX_ROWWISE)
    return e4 ? launch_gemm2<kMxf8, false, false, mxout_code(0, 1)>(qa, qb, K, a, st)
              : launch_gemm2<kMxf8, false, false, mxout_code(1, 1)>(qa, qb, K, a, st);
  if (layout == MX_COLWISE)
    return e4 ? launch_gemm2<kMxf8, false, false, mxout_code(0, 2)>(qa, qb, K, a, st)
              : launch_gemm2<kMxf8, false, false, mxout_code(1, 2)>(qa, qb, K, a, st);
  return e4 ? launch_gemm2<kMxf8, false, false, mxout_code(0, 3)>(qa, qb, K, a, st)
            : launch_gemm2<kMxf8, false, false, mxout_code(1, 3)>(qa, qb, K, a, st);
}

mx_status mx_gemm_mxout(const void* qa, const void* sa, mx_elem ea, const void* qb, const void* sb, mx_elem eb,
                        int64_t M, int64_t N, int64_t K, mx_elem out_elem, void* q_out, void* s_out, int64_t ldq,
                        void* stream) {
  return mx_gemm_mxout_ex(qa, sa, ea, qb, sb, eb, M, N, K, out_elem, MX_ROWWISE, q_out, s_out, ldq, nullptr, nullptr,
                          0, stream);
}

mx_status mx_gemm_grouped(const void* qa, const void* sa, mx_elem ea, const void* qb, const void* sb, mx_elem eb,
                          const int64_t* group_offsets, int64_t groups, int64_t M, int64_t N, int64_t K, void* out,
                          mx_out out_dtype, int64_t ldc, void* stream) {
  if (!qa || !sa || !qb || !sb || !out || !group_offsets) return MX_ERR_INVALID_ARG;
  if (groups < 1 || groups > kMaxGroups) return MX_ERR_INVALID_ARG;
  const bool fp4 = ea == MX_E2M1 && eb == MX_E2M1;   // MXFP4 experts
  if (!gemm_shape_ok(M, N, K, fp4 ? 256 : 128, ldc, out_dtype) || N % 256) return MX_ERR_INVALID_ARG;
  if (groups * N > (1ll << 30)) return MX_ERR_INVALID_ARG;
  if (!aligned(qa, 16) || !aligned(qb, 16) || !aligned(sa, 16) || !aligned(sb, 16) || !aligned(out, 16) ||
      !aligned(group_offsets, 8))
    return MX_ERR_INVALID_ARG;
  if (!fp4 && ((ea != MX_E4M3 && ea != MX_E5M2) || (eb != MX_E4M3 && eb != MX_E5M2))) {
    if (ea == MX_E2M1 || eb == MX_E2M1) return MX_ERR_UNSUPPORTED;   // FP4 x FP8 mixes
    return MX_ERR_INVALID_ARG;
  }
  GemmArgs a{};
  a.sfa = static_cast<const uint8_t*>(sa);
  a.sfb = static_cast<const uint8_t*>(sb);
  a.out = out;
  a.ldc = ldc;
  a.M = static_cast<int>(M);
  a.N = static_cast<int>(N);
  a.K = static_cast<int>(K);
  a.group_off = group_offsets;
  a.groups = static_cast<int>(groups);
  cudaStream_t st = as_stream(stream);
  if (fp4) {
    a.idesc = make_idesc_block_scaled(1u, 1u, 256, 256, 1);
    if (out_dtype == MX_OUT_BF16) return launch_gemm2<kMxf4, true, true>(qa, qb, K / 2, a, st, groups * N);
    return launch_gemm2<kMxf4, false, true>(qa, qb, K / 2, a, st, groups * N);
  }
  a.idesc = make_idesc_block_scaled(static_cast<uint32_t>(ea), static_cast<uint32_t>(eb), 256, 256, 1);
  if (out_dtype == MX_OUT_BF16) return launch_gemm2<kMxf8, true, true>(qa, qb, K, a, st, groups * N);
  return launch_gemm2<kMxf8, false, true>(qa, qb, K, a, st, groups * N);
}

mx_status nvfp4_gemm_grouped(const void* qa, const void* sa, const float* ga, const void* qb, const void* sb,
                             const float* gb, const int64_t* group_offsets, int64_t groups, int64_t M, int64_t N,
                             int64_t K, void* out, mx_out out_dtype, int64_t ldc, void* stream) {
  return nvfp4_gemm_grouped_ex(qa, sa, ga, 0, qb, sb, gb, group_offsets, groups, M, N, K, out, out_dtype, ldc, stream);
}

mx_status nvfp4_gemm_grouped_ex(const void* qa, const void* sa, const float* ga, int ga_per_group, const void* qb,
                                const void* sb, const float* gb, const int64_t* group_offsets, int64_t groups,
                                int64_t M, int64_t N, int64_t K, void* out, mx_out out_dtype, int64_t ldc,
                                void* stream) {
  if (!qa || !sa || !ga || !qb || !sb || !gb || !out || !group_offsets) return MX_ERR_INVALID_ARG;
  if (ga_per_group != 0 && ga_per_group != 1) return MX_ERR_INVALID_ARG;
  if (groups < 1 || groups > kMaxGroups) return MX_ERR_INVALID_ARG;
  if (!gemm_shape_ok(M, N, K, 256, ldc, out_dtype) || N % 256) return MX_ERR_INVALID_ARG;
  if (groups * N > (1ll << 30)) return MX_ERR_INVALID_ARG;
  if (!aligned(qa, 16) || !aligned(qb, 16) || !aligned(sa, 16) || !aligned(sb, 16) || !aligned(out, 16) ||
      !aligned(ga, 4) || !aligned(gb, 4) || !aligned(group_offsets, 8))
    return MX_ERR_INVALID_ARG;
  GemmArgs a{};
  a.sfa = static_cast<const uint8_t*>(sa);
  a.sfb = static_cast<const uint8_t*>(sb);
  a.ga = ga;
  a.gb = gb;
  a.ga_stride = ga_per_group;
  a.out = out;
  a.ldc = ldc;
  a.M = static_cast<int>(M);
  a.N = static_cast<int>(N);
  a.K = static_cast<int>(K);
  a.group_off = group_offsets;
  a.groups = static_cast<int>(groups);
  a.idesc = make_idesc_block_scaled(1u, 1u, 256, 256, 0);
  cudaStream_t st = as_stream(stream);
  if (out_dtype == MX_OUT_BF16) return launch_gemm2<kNvf4, true, true>(qa, qb, K / 2, a, st, groups * N);
  return launch_gemm2<kNvf4, false, true>(qa, qb, K / 2, a, st, groups * N);
}

size_t nvfp4_workspace_bytes(int64_t rows, int64_t cols) {
  (void)rows;
  (void)cols;
  return 16;
}

mx_status mx_scales_from_fp32_blocks(const float* s, int64_t rows, int64_t cols, int block_rows, void* s_e8m0,
                                     void* stream) {
  if (!s || !s_e8m0 || rows <= 0 || cols <= 0 || rows % 128 || cols % 128) return MX_ERR_INVALID_ARG;
  if (block_rows != 1 && block_rows != 128) return MX_ERR_INVALID_ARG;
  if (!aligned(s, 4) || !aligned(s_e8m0, 16)) return MX_ERR_INVALID_ARG;
  dim3 grid;
  if (!quant_grid(rows / 128, cols / 128, &grid)) return MX_ERR_INVALID_ARG;
  pdl_launch(mx_scales_from_blocks_kernel, grid, 128, 0, as_stream(stream), s, rows, cols, block_rows,
                                                                      static_cast<uint8_t*>(s_e8m0));
  return launch_status();
}

namespace {
// One CTA waits, through the bounded wait every kernel of the library uses, on an mbarrier that
// nothing arrives on: the wait runs out after budget_ns, sets the abort flag and its bit in the
// device error word, and the kernel returns.
__global__ void selftest_wait_kernel(unsigned long long budget_ns) {
  pdl_prologue();
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_wait(&bar, 0, &abort_flag, kSiteSelfTest, budget_ns);
}
}  // namespace

mx_status mx_selftest_wait_timeout(int64_t budget_us, void* stream) {
  if (budget_us < 1 || budget_us > 1000000) return MX_ERR_INVALID_ARG;
  pdl_launch(selftest_wait_kernel, 1, 32, 0, as_stream(stream), static_cast<unsigned long long>(budget_us) * 1000ull);
  return launch_status();
}

namespace {
mx_status scale_layout(const void* src, int64_t rows, int64_t nblocks, void* dst, bool to_plain, void* stream) {
  if (!src || !dst || rows <= 0 || nblocks <= 0 || rows % 128 || nblocks % 4) return MX_ERR_INVALID_ARG;
  if (rows > (1ll << 40) / nblocks) return MX_ERR_INVALID_ARG;
  const void* swz = to_plain ? src : dst;
  const void* plain = to_plain ? dst : src;
  if (!aligned(swz, 16) || !aligned(plain, 4)) return MX_ERR_INVALID_ARG;
  const int sms = device_sms();
  if (sms <= 0) return MX_ERR_CUDA;
  const int64_t pieces = rows / 128 * (nblocks / 4) * 32;
  int64_t grid = (pieces + 255) / 256;
  if (grid > 8ll * sms) grid = 8ll * sms;
  const uint8_t* s = static_cast<const uint8_t*>(src);
  uint8_t* d = static_cast<uint8_t*>(dst);
  const dim3 g(static_cast<unsigned>(grid));
  if (to_plain) pdl_launch(scale_layout_kernel<true>, g, 256, 0, as_stream(stream), s, d, rows, nblocks);
  else pdl_launch(scale_layout_kernel<false>, g, 256, 0, as_stream(stream), s, d, rows, nblocks);
  return launch_status();
}
}  // namespace

mx_status mx_unswizzle_scales(const void* s_gemm, int64_t rows, int64_t nblocks, void* s_plain, void* stream) {
  return scale_layout(s_gemm, rows, nblocks, s_plain, true, stream);
}

mx_status mx_swizzle_scales(const void* s_plain, int64_t rows, int64_t nblocks, void* s_gemm, void* stream) {
  return scale_layout(s_plain, rows, nblocks, s_gemm, false, stream);
}

}  // extern "C"

namespace {
// Pass 1 of every NVFP4 quantizer: clear the workspace word, then the global maximum (of the
// transformed values when rht).
mx_status nvfp4_pass1(const uint16_t* x, int64_t rows, int64_t cols, unsigned int* amax, bool rht, uint32_t signs,
                      cudaStream_t st) {
  if (pdl_launch(zero_words_kernel, 1, 256, 0, st, amax, 1) != cudaSuccess) return MX_ERR_CUDA;
  const int sms = device_sms();
  if (sms <= 0) return MX_ERR_CUDA;
  const int64_t nvec = rows * cols / 8;
  int64_t grid1 = (nvec + 255) / 256;
  if (grid1 > 8ll * sms) grid1 = 8ll * sms;
  if (rht) pdl_launch(nvfp4_amax_kernel<true>, static_cast<unsigned>(grid1), 256, 0, st, x, nvec, amax, signs);
  else pdl_launch(nvfp4_amax_kernel<false>, static_cast<unsigned>(grid1), 256, 0, st, x, nvec, amax, 0u);
  return cudaGetLastError() == cudaSuccess ? MX_OK : MX_ERR_CUDA;
}

bool nvfp4_args_ok(const void* x, int64_t rows, int64_t cols, int64_t colmult, const void* q, const void* s,
                   const float* gscale, const void* workspace) {
  if (!x || !q || !s || !gscale || !workspace) return false;
  if (rows <= 0 || cols <= 0 || rows % 128 || cols % colmult) return false;
  if (rows > (1ll << 31) || cols > (1ll << 31)) return false;
  return aligned(x, 16) && aligned(q, 16) && aligned(s, 16) && aligned(gscale, 4) && aligned(workspace, 16);
}
}  // namespace

extern "C" {

mx_status nvfp4_quantize(const void* x, int64_t rows, int64_t cols, void* q_packed, void* s_ue4m3, float* gscale,
                         void* workspace, void* stream) {
  return nvfp4_quantize_ex(x, rows, cols, 0, 0u, nullptr, q_packed, s_ue4m3, gscale, workspace, stream);
}

mx_status nvfp4_quantize_ex(const void* x, int64_t rows, int64_t cols, int use_rht, uint32_t rht_signs,
                            const void* rbits, void* q_packed, void* s_ue4m3, float* gscale, void* workspace,
                            void* stream) {
  if (!nvfp4_args_ok(x, rows, cols, 64, q_packed, s_ue4m3, gscale, workspace)) return MX_ERR_INVALID_ARG;
  if ((use_rht != 0 && use_rht != 1) || rht_signs > 0xFFFFu) return MX_ERR_INVALID_ARG;
  if (rbits && !aligned(rbits, 16)) return MX_ERR_INVALID_ARG;
  cudaStream_t st = as_stream(stream);
  auto* amax = static_cast<unsigned int*>(workspace);
  const auto* xb = static_cast<const uint16_t*>(x);
  const mx_status p1 = nvfp4_pass1(xb, rows, cols, amax, use_rht != 0, rht_signs, st);
  if (p1 != MX_OK) return p1;
  dim3 grid;
  if (!quant_grid(rows / 32, (cols + 127) / 128, &grid)) return MX_ERR_INVALID_ARG;
  auto* q = static_cast<uint8_t*>(q_packed);
  auto* sf = static_cast<uint8_t*>(s_ue4m3);
  const auto* rb = static_cast<const uint8_t*>(rbits);
  // (launched through a function pointer: every parameter is passed, defaults included)
  constexpr const uint8_t* kNoRbits = nullptr;
  constexpr const int64_t* kNoGroups = nullptr;
  if (use_rht && rbits)
    pdl_launch(nvfp4_quantize_kernel<true, true>, grid, 256, 0, st, xb, rows, cols, q, sf, gscale, amax, rht_signs,
               rb, kNoGroups, 1);
  else if (use_rht)
    pdl_launch(nvfp4_quantize_kernel<true, false>, grid, 256, 0, st, xb, rows, cols, q, sf, gscale, amax, rht_signs,
               kNoRbits, kNoGroups, 1);
  else if (rbits)
    pdl_launch(nvfp4_quantize_kernel<false, true>, grid, 256, 0, st, xb, rows, cols, q, sf, gscale, amax, 0u, rb,
               kNoGroups, 1);
  else
    pdl_launch(nvfp4_quantize_kernel<false, false>, grid, 256, 0, st, xb, rows, cols, q, sf, gscale, amax, 0u,
               kNoRbits, kNoGroups, 1);
  return launch_status();
}

mx_status nvfp4_quantize_grouped(const void* x, int64_t rows, int64_t cols, const int64_t* group_offsets,
                                 int64_t groups, void* q_packed, void* s_ue4m3, float* gscale, void* workspace,
                                 void* stream) {
  if (!nvfp4_args_ok(x, rows, cols, 64, q_packed, s_ue4m3, gscale, workspace)) return MX_ERR_INVALID_ARG;
  if (!group_offsets || !aligned(group_offsets, 8) || groups < 1 || groups > kMaxGroups) return MX_ERR_INVALID_ARG;
  cudaStream_t st = as_stream(stream);
  auto* amax = static_cast<unsigned int*>(workspace);
  const auto* xb = static_cast<const uint16_t*>(x);
  const int g = static_cast<int>(groups);
  if (pdl_launch(zero_words_kernel, (g + 255) / 256, 256, 0, st, amax, g) != cudaSuccess) return MX_ERR_CUDA;
  const int sms = device_sms();
  if (sms <= 0) return MX_ERR_CUDA;
  int64_t grid1 = rows / 16;
  if (grid1 > 8ll * sms) grid1 = 8ll * sms;
  pdl_launch(nvfp4_amax_grouped_kernel, static_cast<unsigned>(grid1), 256, 0, st, xb, rows, cols, group_offsets, g,
             amax);
  if (cudaGetLastError() != cudaSuccess) return MX_ERR_CUDA;
  dim3 grid;
  if (!quant_grid(rows / 32, (cols + 127) / 128, &grid)) return MX_ERR_INVALID_ARG;
  pdl_launch(nvfp4_quantize_kernel<false, false, true>, grid, 256, 0, st, xb, rows, cols,
             static_cast<uint8_t*>(q_packed), static_cast<uint8_t*>(s_ue4m3), gscale, amax, 0u,
             static_cast<const uint8_t*>(nullptr), group_offsets, g);
  return launch_status();
}

mx_status nvfp4_quantize_2d(const void* x, int64_t rows, int64_t cols, void* q_row, void* s_row, void* q_col,
                            void* s_col, float* gscale, void* workspace, void* stream) {
  if (!nvfp4_args_ok(x, rows, cols, 128, q_row, s_row, gscale, workspace)) return MX_ERR_INVALID_ARG;
  if (!q_col || !s_col || !aligned(q_col, 16) || !aligned(s_col, 16)) return MX_ERR_INVALID_ARG;
  cudaStream_t st = as_stream(stream);
  auto* amax = static_cast<unsigned int*>(workspace);
  const auto* xb = static_cast<const uint16_t*>(x);
  const mx_status p1 = nvfp4_pass1(xb, rows, cols, amax, false, 0u, st);
  if (p1 != MX_OK) return p1;
  dim3 grid;
  if (!quant_grid(rows / 128, cols / 128, &grid)) return MX_ERR_INVALID_ARG;
  pdl_launch(nvfp4_quantize_2d_kernel, grid, 256, 0, st, xb, rows, cols, static_cast<uint8_t*>(q_row),
                                                 static_cast<uint8_t*>(s_row), static_cast<uint8_t*>(q_col),
                                                 static_cast<uint8_t*>(s_col), gscale, amax);
  return launch_status();
}

mx_status nvfp4_gemm(const void* qa, const void* sa, const float* ga, const void* qb, const void* sb, const float* gb,
                     int64_t M, int64_t N, int64_t K, void* out, mx_out out_dtype, int64_t ldc, void* stream) {
  if (!qa || !sa || !ga || !qb || !sb || !gb || !out) return MX_ERR_INVALID_ARG;
  if (!gemm_shape_ok(M, N, K, 256, ldc, out_dtype)) return MX_ERR_INVALID_ARG;
  if (!aligned(qa, 16) || !aligned(qb, 16) || !aligned(sa, 16) || !aligned(sb, 16) || !aligned(out, 16) ||
      !aligned(ga, 4) || !aligned(gb, 4))
    return MX_ERR_INVALID_ARG;
  GemmArgs a{};
  a.sfa = static_cast<const uint8_t*>(sa);
  a.sfb = static_cast<const uint8_t*>(sb);
  a.ga = ga;
  a.gb = gb;
  a.out = out;
  a.ldc = ldc;
  a.M = static_cast<int>(M);
  a.N = static_cast<int>(N);
  a.K = static_cast<int>(K);
  const bool bn256 = (N % 256) == 0;
  cudaStream_t st = as_stream(stream);
  const bool bf = out_dtype == MX_OUT_BF16;
  const int64_t kb = K / 2;
  if (bn256 && (M % 256) == 0) {
    a.idesc = make_idesc_block_scaled(1u, 1u, 256, 256, 0);
    return bf ? launch_gemm2<kNvf4, true>(qa, qb, kb, a, st) : launch_gemm2<kNvf4, false>(qa, qb, kb, a, st);
  }
  a.idesc = make_idesc_block_scaled(1u, 1u, 128, bn256 ? 256 : 128, 0);
  if (bn256)
    return bf ? launch_gemm<kNvf4, 256, true>(qa, qb, kb, a, st)
              : launch_gemm<kNvf4, 256, false>(qa, qb, kb, a, st);
  return bf ? launch_gemm<kNvf4, 128, true>(qa, qb, kb, a, st) : launch_gemm<kNvf4, 128, false>(qa, qb, kb, a, st);
}

mx_status fp8_blockwise_gemm(const void* qa, const float* sa, const void* qb, const float* sb, int64_t M, int64_t N,
                             int64_t K, void* out, mx_out out_dtype, int64_t ldc, void* stream) {
  if (!qa || !sa || !qb || !sb || !out) return MX_ERR_INVALID_ARG;
  if (!gemm_shape_ok(M, N, K, 128, ldc, out_dtype)) return MX_ERR_INVALID_ARG;
  if (!aligned(qa, 16) || !aligned(qb, 16) || !aligned(sa, 4) || !aligned(sb, 4) || !aligned(out, 16))
    return MX_ERR_INVALID_ARG;
  GemmArgs a{};
  a.dsa = sa;
  a.dsb = sb;
  a.out = out;
  a.ldc = ldc;
  a.M = static_cast<int>(M);
  a.N = static_cast<int>(N);
  a.K = static_cast<int>(K);
  cudaStream_t st = as_stream(stream);
  if (M % 256 == 0 && N % 256 == 0) {  // CTA pairs, 256 x 256 tiles
    a.idesc = make_idesc_f8f6f4(0u, 0u, 256, 256);
    if (out_dtype == MX_OUT_BF16) return launch_ds_gemm2<true>(qa, qb, a, st);
    return launch_ds_gemm2<false>(qa, qb, a, st);
  }
  a.idesc = make_idesc_f8f6f4(0u, 0u, 128, 128);
  if (out_dtype == MX_OUT_BF16) return launch_gemm<kDsF8, 128, true>(qa, qb, K, a, st);
  return launch_gemm<kDsF8, 128, false>(qa, qb, K, a, st);
}

mx_status fp8_blockwise_gemm_grouped(const void* qa, const float* sa, const void* qb, const float* sb,
                                     const int64_t* group_offsets, int64_t groups, int64_t M, int64_t N, int64_t K,
                                     void* out, mx_out out_dtype, int64_t ldc, void* stream) {
  if (!qa || !sa || !qb || !sb || !out || !group_offsets) return MX_ERR_INVALID_ARG;
  if (groups < 1 || groups > kMaxGroups) return MX_ERR_INVALID_ARG;
  if (!gemm_shape_ok(M, N, K, 128, ldc, out_dtype) || N % 256) return MX_ERR_INVALID_ARG;
  if (groups * N > (1ll << 30)) return MX_ERR_INVALID_ARG;
  if (!aligned(qa, 16) || !aligned(qb, 16) || !aligned(sa, 4) || !aligned(sb, 4) || !aligned(out, 16) ||
      !aligned(group_offsets, 8))
    return MX_ERR_INVALID_ARG;
  GemmArgs a{};
  a.dsa = sa;
  a.dsb = sb;
  a.out = out;
  a.ldc = ldc;
  a.M = static_cast<int>(M);
  a.N = static_cast<int>(N);
  a.K = static_cast<int>(K);
  a.group_off = group_offsets;
  a.groups = static_cast<int>(groups);
  a.idesc = make_idesc_f8f6f4(0u, 0u, 256, 256);
  cudaStream_t st = as_stream(stream);
  if (out_dtype == MX_OUT_BF16) return launch_ds_gemm2<true, true>(qa, qb, a, st, groups * N);
  return launch_ds_gemm2<false, true>(qa, qb, a, st, groups * N);
}

mx_status mx_check(void* stream) {
  if (cudaStreamSynchronize(as_stream(stream)) != cudaSuccess) return MX_ERR_CUDA;
  unsigned int word = 0;
  if (cudaMemcpyFromSymbol(&word, g_mx_error_word, sizeof(word)) != cudaSuccess) return MX_ERR_CUDA;
  if (word) {
    const unsigned int zero = 0;
    if (cudaMemcpyToSymbol(g_mx_error_word, &zero, sizeof(zero)) != cudaSuccess) return MX_ERR_CUDA;
    return (word & ~static_cast<unsigned int>(kSiteBadGroups)) ? MX_ERR_TIMEOUT : MX_ERR_INVALID_ARG;
  }
  return MX_OK;
}

}  // extern "C"

// =============================================================================================
// nvfp4_quantize_noalloc: the NVFP4 quantizer for callers that cannot allocate device memory.
//
// nvfp4_quantize needs a small caller-provided workspace for the global amax.  Some callers have
// no way to provide one: a plug-in running inside a host process whose allocator owns all of the
// device memory, or a runtime that must never call cudaMalloc on its launch path because that
// call synchronizes the whole device.  This variant keeps its scratch in the file-scope array
// below, which the library reserves on every GPU it is loaded on, for as long as the process
// lives.  The array holds one partial maximum per band of 16 input rows (16384 bands, 64 KB),
// so inputs may have at most 262144 rows; larger inputs are rejected with MX_ERR_INVALID_ARG.
// =============================================================================================
namespace {
constexpr int64_t kNoAllocBandRows = 16;
constexpr int64_t kNoAllocSlots = 16384;
constexpr int64_t kNoAllocMaxRows = kNoAllocBandRows * kNoAllocSlots;
}  // namespace

// slots [0, kNoAllocSlots): per-band partial maxima (FP32 bits); slot kNoAllocSlots: global amax
static __device__ __align__(256) unsigned int g_nvfp4_noalloc_scratch[kNoAllocSlots + 64];

namespace mxgb {

// One CTA per band of 16 rows: the band's max |x| as FP32 bits.  Writes every slot it owns, so
// nothing in the array has to be cleared between calls.
__global__ void __launch_bounds__(256) nvfp4_band_amax_kernel(const uint16_t* __restrict__ x, int64_t cols,
                                                              unsigned int* __restrict__ partial) {
  pdl_prologue();
  __shared__ uint32_t wmax[8];
  const uint16_t* xb = x + static_cast<int64_t>(blockIdx.x) * kNoAllocBandRows * cols;
  const int64_t nvec = kNoAllocBandRows * cols / 8;
  uint32_t m = 0;
  for (int64_t i = threadIdx.x; i < nvec; i += 256) m = max(m, absmax_bits8(ld_stream_v4(xb + i * 8)));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
  if ((threadIdx.x & 31) == 0) wmax[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int i = 1; i < 8; ++i) m = max(m, wmax[i]);
    partial[blockIdx.x] = m << 16;  // bf16 bits -> FP32 bits
  }
}

// One CTA: maximum over the first `nbands` partial maxima -> *amax_out.
__global__ void __launch_bounds__(1024) nvfp4_amax_finalize_kernel(const unsigned int* __restrict__ partial,
                                                                   int64_t nbands, unsigned int* __restrict__ amax_out) {
  pdl_prologue();
  __shared__ uint32_t wmax[32];
  uint32_t m = 0;
  for (int64_t i = threadIdx.x; i < nbands; i += 1024) m = max(m, partial[i]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
  if ((threadIdx.x & 31) == 0) wmax[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int i = 1; i < 32; ++i) m = max(m, wmax[i]);
    *amax_out = m;
  }
}

}  // namespace mxgb

namespace {
// Device address of the scratch array, looked up once per device with that device current.
unsigned int* noalloc_scratch() {
  static std::mutex mu;
  static unsigned int* addr[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_nvfp4_noalloc_scratch) != cudaSuccess || !p) return nullptr;
    addr[dev] = static_cast<unsigned int*>(p);
  }
  return addr[dev];
}
}  // namespace

extern "C" mx_status nvfp4_quantize_noalloc(const void* x, int64_t rows, int64_t cols, void* q_packed,
                                            void* s_ue4m3, float* gscale, void* stream) {
  if (!x || !q_packed || !s_ue4m3 || !gscale) return MX_ERR_INVALID_ARG;
  if (rows <= 0 || cols <= 0 || rows % 128 || cols % 64) return MX_ERR_INVALID_ARG;
  if (rows > kNoAllocMaxRows || cols > (1ll << 31)) return MX_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(q_packed, 16) || !aligned(s_ue4m3, 16) || !aligned(gscale, 4))
    return MX_ERR_INVALID_ARG;
  unsigned int* scratch = noalloc_scratch();
  if (!scratch) return MX_ERR_CUDA;
  cudaStream_t st = as_stream(stream);
  const int64_t nbands = rows / kNoAllocBandRows;
  pdl_launch(nvfp4_band_amax_kernel, static_cast<unsigned>(nbands), 256, 0, st, static_cast<const uint16_t*>(x), cols,
                                                                         scratch);
  if (cudaGetLastError() != cudaSuccess) return MX_ERR_CUDA;
  pdl_launch(nvfp4_amax_finalize_kernel, 1, 1024, 0, st, scratch, nbands, scratch + kNoAllocSlots);
  if (cudaGetLastError() != cudaSuccess) return MX_ERR_CUDA;
  dim3 grid;
  if (!quant_grid(rows / 32, (cols + 127) / 128, &grid)) return MX_ERR_INVALID_ARG;
  pdl_launch(nvfp4_quantize_kernel<false, false, false>, grid, 256, 0, st, static_cast<const uint16_t*>(x), rows,
             cols, static_cast<uint8_t*>(q_packed), static_cast<uint8_t*>(s_ue4m3), gscale,
             static_cast<const unsigned int*>(scratch + kNoAllocSlots), 0u, static_cast<const uint8_t*>(nullptr),
             static_cast<const int64_t*>(nullptr), 1);
  return launch_status();
}
