// prepass.cuh -- small kernels that run before the pair kernel: the upload of a
// grouped launch's descriptors and the f16 pre-pass of the A operand.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

#include "pair_kernel.cuh"

namespace nf4 {

// ------------------------------------------------------------------ descriptor upload
// Descriptors of a grouped launch travel to the workspace as kernel parameters
// (copied by value at launch, also when the launch is captured in a CUDA graph),
// kDescsPerUpload at a time.
constexpr int kDescsPerUpload = 48;
struct DescChunk {
  ProblemDesc d[kDescsPerUpload];
};
static_assert(sizeof(DescChunk) <= 32000, "kernel parameter limit");

__global__ void upload_descs_kernel(const __grid_constant__ DescChunk chunk, ProblemDesc* dst,
                                    int n) {
  const uint4* src = reinterpret_cast<const uint4*>(&chunk);
  uint4* out = reinterpret_cast<uint4*>(dst);
  const int words = n * static_cast<int>(sizeof(ProblemDesc) / sizeof(uint4));
  for (int i = threadIdx.x; i < words; i += blockDim.x) out[i] = src[i];
}

// ------------------------------------------------------------------ f16 pre-pass
// grad_out [M][N] (fp32 or bf16) -> f16 [M][ldh], ldh = N rounded up to 8:
// the A operand of the pre-converted GEMM variant, with the same rounding the
// converter warps apply (bf16 widened exactly to fp32, then fp32 -> f16 to
// nearest even).  One thread per 16 elements of a row (two 16-byte stores, all
// loads issued before the conversions); columns N..ldh-1 are written as zeros
// (the GEMM's tensor map ends at N and never reads them).  Pure streaming.
//
// A job may also write a column slice of a wider f16 matrix (the fused
// sibling projections: each projection's grad_out goes into its columns of one
// A operand): `width` columns (N rounded up to 8) starting at dst, rows
// `pitch` elements apart.  f16 input is copied as it is.
enum : int { kSrcBF16 = 0, kSrcF32 = 1, kSrcF16 = 2 };
__device__ __forceinline__ uint4 f32x8_to_f16(const float4 a, const float4 b) {
  uint4 h;
  h.x = pack_f16x2(a.x, a.y);
  h.y = pack_f16x2(a.z, a.w);
  h.z = pack_f16x2(b.x, b.y);
  h.w = pack_f16x2(b.z, b.w);
  return h;
}

__device__ __forceinline__ uint4 bf16x8_to_f16(const uint4 w) {
  uint4 h;
  h.x = pack_f16x2(__uint_as_float(w.x << 16), __uint_as_float(w.x & 0xFFFF0000u));
  h.y = pack_f16x2(__uint_as_float(w.y << 16), __uint_as_float(w.y & 0xFFFF0000u));
  h.z = pack_f16x2(__uint_as_float(w.z << 16), __uint_as_float(w.z & 0xFFFF0000u));
  h.w = pack_f16x2(__uint_as_float(w.w << 16), __uint_as_float(w.w & 0xFFFF0000u));
  return h;
}

// One 16-element group (row m, columns c .. c+15 of the width) of the copy.
__device__ __forceinline__ void convert_group(const void* __restrict__ src, int mode,
                                              uint16_t* __restrict__ dst, int N, int width,
                                              int pitch, int64_t m, int c) {
  uint16_t* out = dst + m * pitch + c;
  const bool second = c + 8 < width;  // the group's second 8 columns exist in the copy
  if (mode == kSrcF32) {
    // N % 4 == 0: each 4-column piece is either inside the row or past N.
    const float4* row = reinterpret_cast<const float4*>(static_cast<const float*>(src) + m * N);
    const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
    const int q = c >> 2;
    const float4 a0 = c < N ? __ldcs(row + q) : z;
    const float4 a1 = c + 4 < N ? __ldcs(row + q + 1) : z;
    const float4 a2 = c + 8 < N ? __ldcs(row + q + 2) : z;
    const float4 a3 = c + 12 < N ? __ldcs(row + q + 3) : z;
    *reinterpret_cast<uint4*>(out) = f32x8_to_f16(a0, a1);
    if (second) *reinterpret_cast<uint4*>(out + 8) = f32x8_to_f16(a2, a3);
  } else {
    // N % 8 == 0 and width == N: whole 8-column pieces only.
    const uint4* row = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(src) + m * N);
    const uint4 z = make_uint4(0u, 0u, 0u, 0u);
    const uint4 w0 = __ldcs(row + (c >> 3));
    const uint4 w1 = second ? __ldcs(row + (c >> 3) + 1) : z;
    if (mode == kSrcF16) {
      *reinterpret_cast<uint4*>(out) = w0;
      if (second) *reinterpret_cast<uint4*>(out + 8) = w1;
    } else {
      *reinterpret_cast<uint4*>(out) = bf16x8_to_f16(w0);
      if (second) *reinterpret_cast<uint4*>(out + 8) = bf16x8_to_f16(w1);
    }
  }
}

__global__ void __launch_bounds__(256) to_f16_kernel(const void* __restrict__ src, int f32,
                                                     uint16_t* __restrict__ dst, int M, int N,
                                                     int ldh, unsigned int* __restrict__ flags,
                                                     int nflags) {
  // The GEMM that follows may be scheduled now (it waits for this kernel's
  // results before it reads them).
  griddep_launch_dependents();
  // The split-tile flags of the GEMM that follows start from zero.
  if (blockIdx.x == 0)
    for (int i = threadIdx.x; i < nflags; i += blockDim.x) flags[i] = 0u;
  const int groups = (ldh + 15) >> 4;  // 16-element groups per row
  const int64_t total = static_cast<int64_t>(M) * groups;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t m = i / groups;
    convert_group(src, f32 ? kSrcF32 : kSrcBF16, dst, N, ldh, ldh, m,
                  static_cast<int>(i - m * groups) << 4);
  }
}

// The same pass over several problems of a grouped launch (or the parts of a
// fused call): job j owns the 16-element groups [begin[j], begin[j+1]) of the
// concatenated list.
constexpr int kF16JobsPerLaunch = 64;
struct F16Job {
  const void* src;
  uint16_t* dst;
  int mode;            // kSrcF32, kSrcBF16 or kSrcF16
  int N;               // source columns
  int ldh;             // columns written (N rounded up to 8)
  int pitch;           // destination row pitch (elements)
  int groups_per_row;  // (ldh + 15) / 16
  int64_t begin;
};
struct F16Jobs {
  F16Job job[kF16JobsPerLaunch];
  int64_t end;  // total groups
  int n;
};
static_assert(sizeof(F16Jobs) <= 4096, "kernel parameter size");

__global__ void __launch_bounds__(256) to_f16_group_kernel(const __grid_constant__ F16Jobs jobs) {
  griddep_launch_dependents();
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < jobs.end;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    int lo = 0, hi = jobs.n - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (jobs.job[mid].begin <= i) lo = mid; else hi = mid - 1;
    }
    const F16Job& j = jobs.job[lo];
    const int64_t local = i - j.begin;
    const int64_t m = local / j.groups_per_row;
    convert_group(j.src, j.mode, j.dst, j.N, j.ldh, j.pitch, m,
                  static_cast<int>(local - m * j.groups_per_row) << 4);
  }
}

// ------------------------------------------------------------------ streamed pre-pass
// The f16 pass of a grouped launch, run BESIDE the GEMM instead of before it.
// The GEMM's tiles consume the problems' A operands in order, a few 256-row
// blocks at a time, and is bound by the tensor pipe and its shared-memory
// feed, while the pass is bound by HBM: run together, the pass's traffic fits
// in the bandwidth the GEMM leaves unused.  A block of this kernel (256
// threads, at most 32 registers, no shared memory) fits on an SM next to a
// GEMM CTA (768 threads x at most 72 registers, ~221 KB of shared memory):
// 55,296 + 8,192 of the 65,536 registers.
//
// Work items are slabs of rows of the problems, in the GEMM's order; blocks
// take them through a global counter, so slabs finish roughly in order.  After
// a slab, the block counts it into its 256-row block's `ready` word (release);
// the GEMM's A producer waits for a block's full count (acquire) before its
// first TMA copy from it.  Only one block per SM works: a second one would
// keep the GEMM's CTA off that SM, so it leaves at once.  The source of the
// next rows is prefetched into L2 ahead of the loads, which gives the pass its
// memory-level parallelism without registers or shared memory.
constexpr int kStreamThreads = 256;
// Rows of a slab: at most 64, fewer for wide rows (slab_rows_for), so that a
// 256-row block of a wide problem is spread over many blocks of the pass
// instead of waiting for four long slabs.
constexpr int kSlabMaxRows = 64;
constexpr size_t kSlabTargetBytes = 256u << 10;  // source bytes of a slab, at most (above 8 rows)
constexpr int kStreamMaxJobs = 256;
constexpr int kStreamClaimWords = 256;  // per-SM claim flags (indexed by %smid)
constexpr int kStreamPrefetchAhead = 8;  // loop turns of source prefetched ahead

struct StreamJob {
  const void* src;      // grad_out [M][N]
  uint16_t* dst;        // f16 copy: ldh columns of rows `pitch` elements apart
  unsigned int* ready;  // [ceil(M / 256)] finished slabs per 256-row block
  int mode, M, N, ldh, pitch;
  int item_begin;       // first work item (slab) of this job
  int groups_per_row;   // (ldh + 15) / 16
  int slab_rows;        // rows per slab (divides 256)
};

// Slab rows for a problem whose pass reads `row_bytes` source bytes per row (all
// parts): the largest of 64, 32, 16, 8 whose slab stays within kSlabTargetBytes.
inline int slab_rows_for(size_t row_bytes) {
  int s = kSlabMaxRows;
  while (s > 8 && static_cast<size_t>(s) * row_bytes > kSlabTargetBytes) s >>= 1;
  return s;
}
struct StreamJobs {
  StreamJob job[kStreamMaxJobs];
  unsigned int* next;    // work-item counter, zero at launch
  unsigned int* claims;  // [kStreamClaimWords] per-SM flags, zero at launch
  int n, items;
};
static_assert(sizeof(StreamJobs) <= 32000, "kernel parameter limit");

__global__ void __launch_bounds__(kStreamThreads, 8)
    to_f16_stream_kernel(const __grid_constant__ StreamJobs jobs) {
  // The GEMM may be scheduled now, beside this kernel's blocks.
  griddep_launch_dependents();
  __shared__ int item_s;
  __shared__ int dup_s;
  if (threadIdx.x == 0) {
    const uint32_t sm = sm_id();
    dup_s = sm < static_cast<uint32_t>(kStreamClaimWords) &&
            atomicCAS(jobs.claims + sm, 0u, 1u) != 0u;
  }
  __syncthreads();
  if (dup_s) return;
  for (;;) {
    if (threadIdx.x == 0) item_s = static_cast<int>(atomicAdd(jobs.next, 1u));
    __syncthreads();
    const int item = item_s;
    __syncthreads();  // every thread has read item_s before it is written again
    if (item >= jobs.items) break;
    int lo = 0, hi = jobs.n - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (jobs.job[mid].item_begin <= item) lo = mid; else hi = mid - 1;
    }
    const StreamJob& j = jobs.job[lo];
    const int r0 = (item - j.item_begin) * j.slab_rows;
    const int rows = min(j.slab_rows, j.M - r0);
    const int gpr = j.groups_per_row;
    const int total = rows * gpr;
    // The slab's source is one contiguous run of rows; each loop turn reads
    // about kStreamThreads groups of 16 elements of it.
    const uint32_t esz = j.mode == kSrcF32 ? 4u : 2u;
    const char* base = static_cast<const char*>(j.src) +
                       static_cast<size_t>(r0) * static_cast<size_t>(j.N) * esz;
    const size_t bytes = static_cast<size_t>(rows) * static_cast<size_t>(j.N) * esz;
    const size_t chunk = static_cast<size_t>(kStreamThreads) * 16u * esz;
    if (threadIdx.x == 0) {
      for (int a = 0; a < kStreamPrefetchAhead; ++a) {
        const size_t off = static_cast<size_t>(a) * chunk;
        if (off < bytes)
          prefetch_l2_bulk(base + off, static_cast<uint32_t>(min(chunk, bytes - off)));
      }
    }
    int turn = 0;
    for (int g = threadIdx.x; g < total; g += kStreamThreads, ++turn) {
      if (threadIdx.x == 0) {
        const size_t off = static_cast<size_t>(turn + kStreamPrefetchAhead) * chunk;
        if (off < bytes)
          prefetch_l2_bulk(base + off, static_cast<uint32_t>(min(chunk, bytes - off)));
      }
      const int m = r0 + g / gpr;
      convert_group(j.src, j.mode, j.dst, j.N, j.ldh, j.pitch, m, (g - (m - r0) * gpr) << 4);
    }
    // Every thread's stores are visible device-wide before the slab is counted.
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) red_release_gpu_add(j.ready + (r0 >> 8), 1u);
  }
}

}  // namespace nf4
