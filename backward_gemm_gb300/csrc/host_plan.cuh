// host_plan.cuh -- host side of the pair kernel: tensor-map encoding, argument
// rules, problem descriptors, occupancy, the stream-K split plan, the
// 256/512-token tile rule and the launch.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <climits>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "pair_kernel.cuh"
#include "prepass.cuh"

namespace nf4 {

// ------------------------------------------------------------------ host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

static bool encode_2d(CUtensorMap* map, CUtensorMapDataType type, const void* base,
                      uint64_t inner, uint64_t outer, uint64_t row_bytes, uint32_t box_inner,
                      uint32_t box_outer, CUtensorMapSwizzle swizzle) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, type, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Tile raster (ProblemDesc::row_group): problems with many row blocks and many
// column tiles run in groups of 4 row blocks, column tiles slowest within a
// group; small problems keep the plain order (columns fastest).
static inline int raster_rows(int tiles_m, int tiles_k) {
  return tiles_m >= 8 && tiles_k >= 16 ? 4 : 1;
}

// Argument rules shared by the single and grouped entry points.
static int check_problem(const void* go, int dtype, const float* scales, const uint8_t* data,
                         const float* grad_A, int M, int N, int K) {
  if (dtype != NF4_F32 && dtype != NF4_BF16 && dtype != NF4_F16) return NF4_ERR_INVALID;
  if (M < 0 || N < 0 || K <= 0 || K % 64 != 0) return NF4_ERR_INVALID;
  if (M == 0) return NF4_OK;
  if (grad_A == nullptr) return NF4_ERR_INVALID;
  if (!aligned(grad_A, 16)) return NF4_ERR_ALIGN;
  if (N == 0) return NF4_OK;
  if (go == nullptr || scales == nullptr || data == nullptr) return NF4_ERR_INVALID;
  if (N % (dtype == NF4_F32 ? 4 : 8) != 0) return NF4_ERR_INVALID;
  if (!aligned(go, 16) || !aligned(data, 16) || !aligned(scales, 4)) return NF4_ERR_ALIGN;
  return NF4_OK;
}

// Everything of a descriptor but the grad_out map.
static int fill_desc_rest(ProblemDesc* d, int dtype, const float* scales, const uint8_t* data,
                          float* grad_A, int M, int N, int K, int epi_cols,
                          int rows_per_tile = BMP) {
  const int KB = K / 64;
  d->scale_tma = 0;
  if (KB % 4 == 0 && aligned(scales, 16)) {
    if (!encode_2d(&d->tm_scales, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, scales,
                   static_cast<uint64_t>(KB), static_cast<uint64_t>(N),
                   static_cast<uint64_t>(KB) * 4, 4, BN, CU_TENSOR_MAP_SWIZZLE_NONE))
      return NF4_ERR_CUDA;
    d->scale_tma = 1;
  }
  if (!encode_2d(&d->tm_nf4, CU_TENSOR_MAP_DATA_TYPE_UINT8, data, static_cast<uint64_t>(K / 2),
                 static_cast<uint64_t>(N), static_cast<uint64_t>(K / 2), BKC / 2, BN,
                 CU_TENSOR_MAP_SWIZZLE_64B))
    return NF4_ERR_CUDA;
  if (!encode_2d(&d->tm_out, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, grad_A, static_cast<uint64_t>(K),
                 static_cast<uint64_t>(M), static_cast<uint64_t>(K) * 4,
                 static_cast<uint32_t>(epi_cols), 32,
                 epi_cols == 16 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B))
    return NF4_ERR_CUDA;
  d->scales = scales;
  d->grad_A = grad_A;
  d->M = M;
  d->N = N;
  d->K = K;
  d->dtype = dtype;
  d->tiles_m = (M + rows_per_tile - 1) / rows_per_tile;
  d->tiles_k = (K + BK - 1) / BK;
  d->row_group = raster_rows(d->tiles_m, d->tiles_k);
  d->n_stages = (N + BN - 1) / BN;
  d->tile_begin = 0;
  return NF4_OK;
}

static int fill_desc(ProblemDesc* d, const void* go, int dtype, const float* scales,
                     const uint8_t* data, float* grad_A, int M, int N, int K) {
  std::memset(d, 0, sizeof(*d));
  const bool f32 = dtype == NF4_F32;
  if (!encode_2d(&d->tm_go, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                 go, static_cast<uint64_t>(N), static_cast<uint64_t>(M),
                 static_cast<uint64_t>(N) * (f32 ? 4 : 2), f32 ? 32 : 64, BM,
                 CU_TENSOR_MAP_SWIZZLE_128B))
    return NF4_ERR_CUDA;
  return fill_desc_rest(d, dtype, scales, data, grad_A, M, N, K, LayoutF32::kEpiCols);
}

// Row pitch (elements) and bytes of the f16 copy of an M x N grad_out.
static inline int f16_pitch(int N) { return (N + 7) & ~7; }
static inline size_t f16_bytes(int M, int N) {
  return sizeof(uint16_t) * static_cast<size_t>(M) * static_cast<size_t>(f16_pitch(N));
}

// Descriptor of the pre-converted variant: the A map reads the f16 copy (box
// 64 columns x 128 rows, 128-byte swizzle = the K-major A operand layout).
static int fill_desc_pre(ProblemDesc* d, const uint16_t* go_f16, const float* scales,
                         const uint8_t* data, float* grad_A, int M, int N, int K,
                         int rows_per_tile = LayoutPreA::kRowsPerTile) {
  std::memset(d, 0, sizeof(*d));
  if (!encode_2d(&d->tm_go, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, go_f16, static_cast<uint64_t>(N),
                 static_cast<uint64_t>(M), static_cast<uint64_t>(f16_pitch(N)) * 2, BN, BM,
                 CU_TENSOR_MAP_SWIZZLE_128B))
    return NF4_ERR_CUDA;
  // dtype is not read by this variant (its A operand is f16 already).
  return fill_desc_rest(d, NF4_BF16, scales, data, grad_A, M, N, K,
                        rows_per_tile == LayoutPreA2::kRowsPerTile ? LayoutPreA2::kEpiCols
                                                                   : LayoutPreA::kEpiCols,
                        rows_per_tile);
}

// Descriptor of the forward product C[M x N] = A[M x K] @ dequant(B_nf4[K x N])
// on the pre-converted kernel: the A map reads the f16 copy of A (box 64
// columns k x 128 rows), the NF4 map boxes 128 rows n x 32 bytes (one 64-k
// block), the output map is C.  The block scales are loaded by the converters.
static int fill_desc_fwd(ProblemDesc* d, const uint16_t* a_f16, const float* scales,
                         const uint8_t* data, float* C, int M, int N, int K, int rows_per_tile) {
  std::memset(d, 0, sizeof(*d));
  const int epi_cols = rows_per_tile == LayoutPreA2::kRowsPerTile ? LayoutPreA2::kEpiCols
                                                                  : LayoutPreA::kEpiCols;
  if (!encode_2d(&d->tm_go, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, a_f16, static_cast<uint64_t>(K),
                 static_cast<uint64_t>(M), static_cast<uint64_t>(f16_pitch(K)) * 2, BN, BM,
                 CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_2d(&d->tm_nf4, CU_TENSOR_MAP_DATA_TYPE_UINT8, data, static_cast<uint64_t>(K / 2),
                 static_cast<uint64_t>(N), static_cast<uint64_t>(K / 2), BN / 2, BKC,
                 CU_TENSOR_MAP_SWIZZLE_NONE) ||
      !encode_2d(&d->tm_out, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, C, static_cast<uint64_t>(N),
                 static_cast<uint64_t>(M), static_cast<uint64_t>(N) * 4,
                 static_cast<uint32_t>(epi_cols), 32,
                 epi_cols == 16 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B))
    return NF4_ERR_CUDA;
  d->scales = scales;
  d->grad_A = C;
  d->M = M;
  d->N = N;
  d->K = K;
  d->dtype = NF4_BF16;  // not read by this variant
  d->tiles_m = (M + rows_per_tile - 1) / rows_per_tile;
  d->tiles_k = (N + BK - 1) / BK;
  d->row_group = raster_rows(d->tiles_m, d->tiles_k);
  d->n_stages = K / BN;
  d->tile_begin = 0;
  d->scale_tma = 0;
  d->fwd = 1;
  return NF4_OK;
}

static int sm_count(int* out) {
  static int cached[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return NF4_ERR_CUDA;
  if (cached[dev] == 0) {
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        sms <= 0)
      return NF4_ERR_CUDA;
    cached[dev] = sms;
  }
  *out = cached[dev];
  return NF4_OK;
}

static int launch_to_f16(const void* go, int dtype, uint16_t* dst, int M, int N,
                         unsigned int* flags, int nflags, cudaStream_t stream) {
  int sms = 0;
  const int rc = sm_count(&sms);
  if (rc != NF4_OK) return rc;
  // One 16-element group per thread; the grid covers all of them in one pass
  // up to 64 resident blocks' worth per SM, beyond that threads loop.
  const int64_t work = static_cast<int64_t>(M) * ((f16_pitch(N) + 15) >> 4);
  const int64_t blocks = std::min<int64_t>((work + 255) / 256, static_cast<int64_t>(sms) * 64);
  to_f16_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
      go, dtype == NF4_F32 ? 1 : 0, dst, M, N, f16_pitch(N), flags, nflags);
  return cudaGetLastError() == cudaSuccess ? NF4_OK : NF4_ERR_CUDA;
}

// The grouped f16 pass over up to kF16JobsPerLaunch jobs.
static int launch_f16_jobs(const F16Jobs& jobs, cudaStream_t stream) {
  int sms = 0;
  const int rc = sm_count(&sms);
  if (rc != NF4_OK) return rc;
  const int64_t blocks = std::min<int64_t>((jobs.end + 255) / 256, static_cast<int64_t>(sms) * 64);
  to_f16_group_kernel<<<static_cast<unsigned>(std::max<int64_t>(blocks, 1)), 256, 0, stream>>>(jobs);
  return cudaGetLastError() == cudaSuccess ? NF4_OK : NF4_ERR_CUDA;
}

// Largest number of pairs of CTAs of kernel configuration L that fit on the
// current device at once (also sets the kernel's shared-memory limit).
template <class L>
static int max_clusters(int* out) {
  static int cached[64] = {};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return NF4_ERR_CUDA;
  std::lock_guard<std::mutex> lock(mu);
  if (cached[dev] == 0) {
    if (cudaFuncSetAttribute(bwd_a_kernel<L>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             L::kSmemBytes) != cudaSuccess)
      return NF4_ERR_CUDA;
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return NF4_ERR_CUDA;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(static_cast<unsigned>(sms & ~1), 1, 1);
    cfg.blockDim = dim3(L::kThreads, 1, 1);
    cfg.dynamicSmemBytes = L::kSmemBytes;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int clusters = 0;
    if (cudaOccupancyMaxActiveClusters(&clusters, bwd_a_kernel<L>, &cfg) != cudaSuccess ||
        clusters <= 0)
      clusters = sms / 2;
    cached[dev] = clusters;
  }
  *out = cached[dev];
  return NF4_OK;
}

// Launch over `total_tiles` tiles; sk == nullptr: all tiles whole, else the
// split described by *sk (planned for this device's pair count).
// pdl: the launch directly follows to_f16_kernel on the stream and may start
// while that kernel finishes (programmatic stream serialization).
template <class L>
static int launch_layout(const ProblemDesc& single, const ProblemDesc* batch, int count,
                         int total_tiles, const SkArgs* sk_in, cudaStream_t stream,
                         bool pdl = false) {
  int maxc = 0;
  const int rc = max_clusters<L>(&maxc);
  if (rc != NF4_OK) return rc;
  SkArgs sk;
  std::memset(&sk, 0, sizeof(sk));
  sk.dp_tiles = total_tiles;
  int clusters = std::min(total_tiles, maxc);
  if (sk_in != nullptr && sk_in->sk_tiles > 0) {
    sk = *sk_in;
    clusters = maxc;
  }
  if (sk_in != nullptr) sk.streamed = sk_in->streamed;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3(static_cast<unsigned>(2 * clusters), 1, 1);
  cfg.blockDim = dim3(L::kThreads, 1, 1);
  cfg.dynamicSmemBytes = L::kSmemBytes;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 2 : 1;
  if (cudaLaunchKernelEx(&cfg, bwd_a_kernel<L>, single, batch, count, sk) != cudaSuccess)
    return NF4_ERR_CUDA;
  return launch_status();
}

// all_bf16: every problem of the launch has bf16 grad_out (the deeper-ring
// layout only has room for bf16 raw stages).
static int launch(const ProblemDesc& single, const ProblemDesc* batch, int count, int total_tiles,
                  bool all_bf16, cudaStream_t stream) {
  return all_bf16 ? launch_layout<LayoutBF16>(single, batch, count, total_tiles, nullptr, stream)
                  : launch_layout<LayoutF32>(single, batch, count, total_tiles, nullptr, stream);
}


// Workspace of nf4_backward_a_ws: the f16 copy of grad_out, then (optional)
// the split-tile flags and partial sums for `pairs` pairs of CTAs.
// Per pair: 2 CTAs x up to 2 M-blocks x 128 x 256 fp32.
constexpr size_t kPartialBytes = static_cast<size_t>(2) * 2 * BM * BK * sizeof(float);  // 512 KiB
static inline size_t round256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }
static inline size_t sk_bytes(int pairs) {
  return round256(sizeof(unsigned int) * static_cast<size_t>(pairs)) +
         kPartialBytes * static_cast<size_t>(pairs);
}

// Split plan for T tiles of S stages over `pairs` pairs: whole waves stay whole;
// the last, partial wave is split by stages when that saves every pair at
// least kSplitMinSaving stages of the wave (S - rem * S / pairs).  A split
// tile costs an extra partial-sum epilogue and a dependent finishing epilogue
// (measured on GB300: worth roughly 30 stages of 64 on the critical path), so
// smaller savings are not taken.
constexpr int kSplitMinSaving = 40;
static void plan_split(int T, int S, int pairs, SkArgs* sk) {
  sk->dp_tiles = T;
  sk->sk_tiles = 0;
  sk->stages = S;
  if (pairs <= 1 || S <= 1) return;
  const int rem = T % pairs;
  if (rem == 0) return;
  if (static_cast<int64_t>(S) * (pairs - rem) < static_cast<int64_t>(kSplitMinSaving) * pairs)
    return;
  sk->dp_tiles = T - rem;
  sk->sk_tiles = rem;
}

// 256- or 512-token pair tiles for the pre-converted kernel.  A 512-token
// stage issues 8 MMAs against one dequantised B^T stage; measured on GB300 it
// takes ~1.4-1.5x a 256-token stage, and a 512-token tile's epilogue does not
// overlap the next tile.  512-token tiles were faster on every measured shape
// with at least 8 stages and at least half a wave of them (down/up/o/gate at
// M = 4096, 2048 x 4096 x 4096, the 8191-token shapes, also against the split
// 256-token schedule); slower on q_proj (24 such tiles for 76 pairs) and on
// N = 256 (4 stages).
static std::atomic<int> g_tile_rows{0};  // 0: by the rule below; 256 or 512: forced

static bool tiles512_rule(int64_t tiles512, int S, int pairs) {
  return S >= 8 && pairs > 0 && 2 * tiles512 >= pairs;
}

static bool use_tiles512(int M, int N, int K, int pairs, bool /*can_split*/) {
  const int forced = g_tile_rows.load();
  if (forced != 0) return forced == 512;
  if (M <= 256) return false;
  const int64_t T2 = static_cast<int64_t>((M + 511) / 512) * ((K + BK - 1) / BK);
  return tiles512_rule(T2, (N + BN - 1) / BN, pairs);
}

}  // namespace nf4
