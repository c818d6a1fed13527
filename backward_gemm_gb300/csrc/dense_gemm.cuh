// dense_gemm.cuh -- the dense weight gradient of a matrix product on tcgen05:
//
//     grad_B[K x N] = A[M x K]^T @ grad_C[M x N]
//
// (page "trueno-gpu 0.4.17 -- src/kernels/backward/mod.rs": the backward
// module's GEMM kernels give the gradients of both operands of C = A @ B;
// GemmBackwardBKernel takes a_ptr and writes grad_b_ptr.)  Next to a frozen
// NF4 base weight this is the gradient of the trainable 16-bit weights (LoRA
// adapters, or any layer trained in full): the contraction runs over the
// tokens M, both operands are 16-bit (bf16 or f16, the same for both) and the
// products are summed in fp32 by the tensor cores.
//
// Both operands are row-major with the tokens as rows, so both are MN-major
// for the MMA (the output dimension contiguous, the contraction strided): a
// TMA box of 64 output indices (128 bytes, 128-byte swizzle) by 64 tokens is
// exactly one 64-wide atom column of that layout, 8 tokens per 1 KB atom.  No
// element is converted or reordered on the way, so the kernel is the pair
// MMA fed by TMA alone:
//
//   pair tile   256 rows k x 256 columns n, a cluster of two CTAs, MMA
//               cta_group::2 M = 256, N = 256, K = 16; CTA r loads A's columns
//               k = 128r .. 128r + 127 of the tile (its half of the M side) and
//               grad_C's columns n = 128r .. (its half of the N side)
//   stage       64 tokens: two 8 KB boxes of each operand per CTA (32 KB), 4 MMAs
//   warp 4      TMA producer: lanes 0-3 issue one box each; both CTAs' copies
//               complete on the leader's barrier
//   warp 5      TMEM allocation; in CTA 0 the MMA issuer, double-buffered
//               accumulator (2 x 256 columns)
//   warps 0-3   epilogue: tcgen05.ld, 64-byte-swizzled staging, TMA store
//               (clipped at K and N)
//
// When the tiles are too few to give every pair of SMs work, the tokens are
// cut into `splits` equal runs: split s of a tile writes its fp32 partial sum
// into slice s of a workspace, and a second kernel adds the slices in order s =
// 0, 1, ... (a fixed order: results do not depend on timing).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "nf4_common.h"
#include "ptx.cuh"

namespace nf4 {
namespace dense {

constexpr int kRowsCta = 128;             // output rows per CTA (MMA M = 256 per pair)
constexpr int kTileK = 2 * kRowsCta;      // output rows per pair tile
constexpr int kTileN = 256;               // output columns per pair tile (MMA N)
constexpr int kTok = 64;                  // tokens per stage (4 MMA K-steps of 16)
constexpr int kStages = 6;
constexpr int kBox = 64 * kTok * 2;       // 8 KB: 64 output indices x 64 tokens
constexpr int kStageBytes = 4 * kBox;     // A: 2 boxes, grad_C: 2 boxes
constexpr int kEpiWarps = 4;
constexpr int kEpiCols = 16;              // fp32 columns per TMEM load / TMA store
constexpr int kEpiBuf = 32 * kEpiCols * 4;
constexpr int kProducerWarp = 4;
constexpr int kMmaWarp = 5;
constexpr int kThreads = 6 * 32;
constexpr uint32_t kTmemCols = 2 * kTileN;

constexpr int kEpiOff = kStages * kStageBytes;
constexpr int kBarOff = kEpiOff + kEpiWarps * 2 * kEpiBuf;
// full[kStages], empty[kStages], tmem_full[2], tmem_empty[2], mma_done
constexpr int kNumBars = 2 * kStages + 5;
constexpr int kMiscOff = kBarOff + kNumBars * 8;  // TMEM address, abort flag
constexpr int kSmemBytes = kMiscOff + 16 + 1024;  // + alignment slack
static_assert(kSmemBytes <= 232448, "shared memory budget");

struct Args {
  CUtensorMap tm_a;    // A [M][K], box 64 k x 64 tokens, 128-byte swizzle
  CUtensorMap tm_c;    // grad_C [M][N], box 64 n x 64 tokens, 128-byte swizzle
  CUtensorMap tm_out;  // grad_B [K][N] fp32, or the split workspace [splits * Kp][N]
  int tiles_k, tiles_n, splits, stages;  // stages: 64-token stages of the whole M
  int items;           // tiles_k * tiles_n * splits
  int kp;              // rows per workspace slice (tiles_k * 256); 0 without a split
  uint32_t idesc;      // MMA instruction descriptor (f16 or bf16, both operands MN-major)
};

// Item i: tile t = i % tiles (columns of n fastest, so pairs running at the
// same time share A's row block), split s = i / tiles over the tokens.
struct Item {
  int tk, tn, s, st0, st1;  // tile, split, stages [st0, st1)
};

__device__ __forceinline__ Item item_of(const Args& a, int i) {
  Item w;
  const int tiles = a.tiles_k * a.tiles_n;
  const int t = i % tiles;
  w.s = i / tiles;
  w.tk = t / a.tiles_n;
  w.tn = t % a.tiles_n;
  w.st0 = static_cast<int>(static_cast<int64_t>(a.stages) * w.s / a.splits);
  w.st1 = static_cast<int>(static_cast<int64_t>(a.stages) * (w.s + 1) / a.splits);
  return w;
}

__global__ void __launch_bounds__(kThreads, 1) backward_b_kernel(const __grid_constant__ Args a) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  const uint32_t sbase = smem_addr(smem);
  const uint32_t rank = cluster_ctarank();
  const int pair = static_cast<int>(blockIdx.x >> 1);
  const int npairs = static_cast<int>(gridDim.x >> 1);
  const uint32_t bar0 = sbase + kBarOff;
  auto full = [&](uint32_t i) { return bar0 + 8u * i; };
  auto empty = [&](uint32_t i) { return bar0 + 8u * (kStages + i); };
  auto tmem_full = [&](uint32_t i) { return bar0 + 8u * (2 * kStages + i); };
  auto tmem_empty = [&](uint32_t i) { return bar0 + 8u * (2 * kStages + 2 + i); };
  const uint32_t mma_done = bar0 + 8u * (2 * kStages + 4);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kMiscOff);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kMiscOff + 4);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 32) {
    tma_prefetch_desc(&a.tm_a);
    tma_prefetch_desc(&a.tm_c);
    tma_prefetch_desc(&a.tm_out);
  }
  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(full(i), 1);   // CTA 0's producer registers both CTAs' bytes
      mbar_init(empty(i), 1);  // the MMA commit (multicast to both CTAs)
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(tmem_full(i), 1);
      mbar_init(tmem_empty(i), 2 * kEpiWarps);  // epilogues of both CTAs (used in CTA 0)
    }
    mbar_init(mma_done, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc_pair(smem_addr(tmem_slot), kTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // both CTAs' barriers are initialised before any remote arrive or copy
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ TMA producer
    // Lane b issues box b of every stage: 0-1 A (k offsets 0, 64 of this CTA's
    // 128 rows), 2-3 grad_C (n offsets 0, 64 of this CTA's 128 columns).
    const uint32_t full_leader0 = mapa_shared(full(0), 0);
    uint32_t it = 0;
    bool ok = true;
    for (int i = pair; ok && i < a.items; i += npairs) {
      const Item w = item_of(a, i);
      for (int st = w.st0; st < w.st1; ++st, ++it) {
        const uint32_t slot = it % kStages;
        bool free_slot = true;
        if (lane == 0)
          free_slot = mbar_wait_cluster(empty(slot), ((it / kStages) & 1u) ^ 1u, abort_flag);
        if (!__shfl_sync(0xFFFFFFFFu, free_slot, 0)) {
          ok = false;
          break;
        }
        if (lane < 4) {
          if (rank == 0 && lane == 0) mbar_arrive_expect_tx(full(slot), 2u * kStageBytes);
          const bool is_a = lane < 2;
          const int x = is_a ? w.tk * kTileK + static_cast<int>(rank) * kRowsCta + 64 * lane
                             : w.tn * kTileN + static_cast<int>(rank) * (kTileN / 2) + 64 * (lane - 2);
          tma_load_2d_pair(sbase + slot * kStageBytes + lane * kBox, is_a ? &a.tm_a : &a.tm_c, x,
                           st * kTok, full_leader0 + 8u * slot);
        }
        __syncwarp();
      }
    }
    if (lane == 0 && ok) {
      // The last commits into this CTA's empty barriers (which also mean that
      // the last copies landed: their MMAs read them) arrive before exit.
      for (uint32_t i = (it > kStages ? it - kStages : 0u); i < it; ++i)
        mbar_wait_cluster(empty(i % kStages), (i / kStages) & 1u, nullptr);
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer (CTA 0)
    if (rank == 0) {
      // A and grad_C slots: MN-major, 128-byte swizzle, the second 64-wide atom
      // column 8 KB on (LBO), 8-token atoms 1 KB apart (SBO); one K-step of
      // 16 tokens is 2 KB further.
      const uint64_t a_desc0 = smem_desc_sw128(sbase, kBox, 1024);
      const uint64_t c_desc0 = smem_desc_sw128(sbase + 2 * kBox, kBox, 1024);
      constexpr uint64_t kStep = 2048 >> 4;
      uint32_t it = 0, lt = 0;
      bool ok = true;
      for (int i = pair; ok && i < a.items; i += npairs, ++lt) {
        const Item w = item_of(a, i);
        const uint32_t acc = lt & 1u;
        if (!__all_sync(0xFFFFFFFFu,
                        mbar_wait_cluster(tmem_empty(acc), ((lt >> 1) & 1u) ^ 1u, abort_flag))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem_base + acc * kTileN;
        for (int st = w.st0; st < w.st1; ++st, ++it) {
          const uint32_t slot = it % kStages;
          // The copies' completion on the barrier makes the operands visible to
          // the MMA (both in the async proxy): no tcgen05 fence per stage.
          if (!__all_sync(0xFFFFFFFFu,
                          mbar_wait_cluster(full(slot), (it / kStages) & 1u, abort_flag))) {
            ok = false;
            break;
          }
          const uint64_t off = static_cast<uint64_t>((slot * kStageBytes) >> 4);
          if (elect_one()) {
#pragma unroll
            for (int k = 0; k < 4; ++k)
              tc_mma_f16_pair(d, a_desc0 + off + k * kStep, c_desc0 + off + k * kStep, a.idesc,
                              (st != w.st0 || k > 0) ? 1u : 0u);
            tc_commit_pair(empty(slot), 0x3);
          }
          __syncwarp();
        }
        if (!ok) break;
        if (elect_one()) tc_commit_pair(tmem_full(acc), 0x3);
        __syncwarp();
      }
      // No MMA may still be writing TMEM (of either CTA) when it is released.
      if (elect_one()) tc_commit_pair(mma_done, 0x1);
      __syncwarp();
      mbar_wait(mma_done, 0, nullptr);
      if (ok) {
        for (uint32_t l = (lt > 2 ? lt - 2 : 0u); l < lt; ++l)
          mbar_wait_cluster(tmem_empty(l & 1u), (l >> 1) & 1u, nullptr);
      }
    }
    __syncwarp();
  } else if (warp < kEpiWarps) {
    // ------------------------------------------------------------ epilogue
    const uint32_t tmem_empty_leader0 = mapa_shared(tmem_empty(0), 0);
    uint8_t* const buf0 = smem + kEpiOff + warp * 2 * kEpiBuf;
    // Row `lane` of a 32-row chunk, 64-byte rows: 16-byte piece q at q ^ ((r / 2) % 4),
    // the layout the 64-byte-swizzled TMA store reads.
    const uint32_t sw = (static_cast<uint32_t>(lane) >> 1) & 3u;
    uint32_t lt = 0;
    int seq = 0;
    for (int i = pair; i < a.items; i += npairs, ++lt) {
      const Item w = item_of(a, i);
      const uint32_t acc = lt & 1u;
      if (!__all_sync(0xFFFFFFFFu, mbar_wait_cluster(tmem_full(acc), (lt >> 1) & 1u, abort_flag)))
        break;
      tc_fence_after();
      const int row = (a.kp > 0 ? w.s * a.kp : 0) + w.tk * kTileK +
                      static_cast<int>(rank) * kRowsCta + warp * 32;
      const uint32_t taddr = tmem_base + acc * kTileN + (static_cast<uint32_t>(warp * 32) << 16);
#pragma unroll 1
      for (int c = 0; c < kTileN / kEpiCols; ++c, ++seq) {
        uint32_t r[kEpiCols];
        tmem_ld_cols<kEpiCols>(taddr + c * kEpiCols, r);
        tmem_wait_ld();
        uint8_t* buf = buf0 + (seq & 1) * kEpiBuf;
        if (lane == 0) bulk_wait_read<1>();  // the store that last read this buffer is done
        __syncwarp();
#pragma unroll
        for (int q = 0; q < kEpiCols / 4; ++q)
          *reinterpret_cast<uint4*>(buf + lane * (kEpiCols * 4) + ((static_cast<uint32_t>(q) ^ sw) << 4)) =
              make_uint4(r[4 * q], r[4 * q + 1], r[4 * q + 2], r[4 * q + 3]);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          tma_store_2d(&a.tm_out, w.tn * kTileN + c * kEpiCols, row, smem_addr(buf));
          bulk_commit();
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (rank == 0) mbar_arrive(tmem_empty(acc));
        else mbar_arrive_remote(tmem_empty_leader0 + 8u * acc);
      }
    }
    if (lane == 0) bulk_wait<0>();
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();  // the leader's MMAs are done and no remote arrive is in flight
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, kTmemCols);
  }
  // After a wait gave up, copies of the peer CTA that complete on this CTA's
  // barriers, or this CTA's own copies that complete on the leader's, may
  // still be in flight: stay resident a bounded time so that they land first.
  if (threadIdx.x == 0 && (*abort_flag != 0 || *(volatile unsigned int*)&g_status != 0)) {
    const long long t0 = clock64();
    while (clock64() - t0 < 4000000) {
    }
  }
}

// grad_B[k][n] = sum over s = 0, 1, ... of slice s of the workspace (rows kp
// apart); N % 4 == 0, so each thread adds float4 columns in a fixed order.
__global__ void __launch_bounds__(256) reduce_splits_kernel(const float* __restrict__ ws,
                                                            float* __restrict__ out, int splits,
                                                            int K, int N, int kp) {
  const int n4 = N >> 2;
  const int64_t total = static_cast<int64_t>(K) * n4;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t k = i / n4;
    const int64_t q = i - k * n4;
    float4 acc = __ldcs(reinterpret_cast<const float4*>(ws + k * N) + q);
    for (int s = 1; s < splits; ++s) {
      const float4 v =
          __ldcs(reinterpret_cast<const float4*>(ws + (static_cast<int64_t>(s) * kp + k) * N) + q);
      acc.x += v.x;
      acc.y += v.y;
      acc.z += v.z;
      acc.w += v.w;
    }
    __stcs(reinterpret_cast<float4*>(out + k * N) + q, acc);
  }
}

}  // namespace dense
}  // namespace nf4
