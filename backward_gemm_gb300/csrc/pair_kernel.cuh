// pair_kernel.cuh -- the persistent tcgen05 pair kernel of the NF4-dequant-fused
// backward-A GEMM (device code and the structures it shares with the host).
//
//     grad_A[M x K] = grad_out[M x N] @ dequant(B_nf4[K x N])^T
//
// (page "aprender-gpu 0.32.0 -- src/kernels/backward/nf4_tensor_core.rs",
// struct doc comment and build_ptx phases 1-4.)  That page's kernel gives one
// warp a 16x16 output tile and runs WMMA 16x16x16 over N; here the same
// arithmetic runs as a persistent, warp-specialised kernel on pairs of SMs:
//
//   pair tile   256 (or 512: two M-blocks) tokens x 256 output columns k,
//               computed by a cluster of two CTAs with tcgen05.mma.cta_group::2
//               (M=256, N=256, K=16).  CTA r of the pair holds grad_out rows
//               128r..128r+127 of each M-block (the A operand) and dequantises
//               B^T for output columns 128r..128r+127 (its half of the B
//               operand); the MMA reads both halves, so each SM dequantises
//               only half of what a single-CTA tile would need.  The shared
//               dimension N is consumed 64 at a time (4 MMAs per M-block).
//   warp 4      raw producer (each CTA): the NF4 bytes (64 rows n x 64 bytes =
//               128 k, 64-byte swizzle) and the stage's block scales, plus
//               grad_out (fp32 or bf16 boxes, 128-byte swizzle) in the variants
//               that convert it in shared memory, into a ring of raw stages
//   warp 23     pre-converted variant: copies each stage's f16 A operand (made
//               by the f16 pre-pass) with TMA into a ring of A slots
//   warps 6-21  converters, two groups of 8 warps that take alternate stages:
//               NF4 codes x block scale -> f16 into the MN-major B^T operand
//               (one 64-k NF4 block is one 128-byte swizzle row), and grad_out
//               -> f16 into the K-major A operand where it is not pre-converted
//   warp 5      allocates 512 TMEM columns in both CTAs; in CTA 0 one elected
//               lane of the converged warp issues the pair MMAs into a
//               double-buffered fp32 accumulator (2 x 256 columns; 512-token
//               tiles use both as one) and commits to barriers of both CTAs.
//               CTA 1's converter warps signal a finished stage to CTA 0 with
//               16-byte bulk copies that complete on CTA 0's operand barrier
//   warp 22     CTA 0: waits on the operand barriers and publishes each ready
//               stage in a shared-memory word the MMA warp polls
//   warps 0-3   epilogue (each CTA): tcgen05.ld of a 32-lane quarter, staged
//               through shared memory (double-buffered, or a whole M-block in
//               the idle rings) and written with TMA stores, which clip rows >=
//               M and columns >= K; overlaps the next tile's main loop when the
//               accumulator is double-buffered
//
// Out-of-range operands contribute 0 (page above, "PHASE 1"/"PHASE 2": zero the
// out-of-bounds elements): TMA fills rows >= M and columns >= N of grad_out
// with zeros, and the scale of every column n >= N is taken as 0.
//
// The same kernel serves one problem (descriptor passed as a kernel parameter)
// and a grouped launch over many projections (descriptors in a caller-owned
// device workspace, tiles of all problems flattened into one list); a single
// problem's last partial wave of tiles may be split by stages over all pairs
// (stream-K, partial sums added in a fixed order).  A per-problem flag turns
// the pre-converted variant around for the forward product C = A @ dequant(B)
// (contracted over K; the dequantised weight becomes a K-major B operand).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <climits>
#include <cstdint>

#include "nf4_common.h"
#include "nf4_dequant.cuh"
#include "ptx.cuh"
#include "nf4_trace.cuh"

namespace nf4 {

// ------------------------------------------------------------------ geometry
constexpr int BM = 128;        // tokens per CTA (half of the pair's MMA M = 256)
constexpr int BMP = 2 * BM;    // tokens per pair tile
constexpr int BK = 256;        // output columns k per pair tile (MMA N)
constexpr int BKC = BK / 2;    // output columns whose B^T one CTA dequantises
constexpr int BN = 64;         // shared-dimension slice per stage (4 x MMA K=16)

constexpr int kEpiWarps = 4;
constexpr int kProducerWarp = 4;
constexpr int kMmaWarp = 5;
constexpr int kConvWarp0 = 6;
constexpr int kConvGroups = 2;   // group g converts the stages it with it % 2 == g
constexpr int kGroupWarps = 8;   // warps per group (256 threads)
constexpr int kConvWarps = kConvGroups * kGroupWarps;
constexpr int kWatchWarp = kConvWarp0 + kConvWarps;       // 22

constexpr int kGoBoxBytes = BM * 128;                  // one 128-byte-wide box of 128 rows
constexpr int kNf4Bytes = BN * (BKC / 2);              // 64 rows n x 64 bytes
constexpr int kScaleBytes = BN * 16;                   // 64 rows n x 4 block scales
constexpr int kABytes = BM * BN * 2;                   // 16 KB f16
constexpr int kBBytes = BKC * BN * 2;                  // 16 KB f16
constexpr int kOpBytes = kABytes + kBBytes;            // 32 KB
constexpr int kEpiBufs = 2;  // staging buffers per epilogue warp: a store drains while the next fills
constexpr uint32_t kSigBytes = 16;
constexpr long long kAbortLingerCycles = 4000000;  // ~2 ms: far longer than a copy's latency
constexpr uint32_t kTmemCols = 2 * BK;

// Shared-memory layout of one kernel configuration: RS raw stages holding GOB
// bytes of grad_out, the NF4 bytes and the stage's block scales, OS operand
// stages, the epilogue staging, barriers and flags.  bf16 grad_out needs half the raw bytes of fp32, which
// buys a deeper ring on both sides.
//
// RA > 0 selects the pre-converted variant: grad_out was rounded to f16 by a
// separate pass, and a TMA copy writes each stage's A operand straight into a
// ring of RA A slots (no raw grad_out, no converter work on A); the operand
// slots then hold B^T only.
template <int RS, int OS, int GOB, int RA = 0, int EC = 16, int MB = 1>
struct Layout {
  static constexpr bool kPreA = RA > 0;
  // M-blocks of 256 tokens per pair tile.  MB = 2 (pre-converted variant
  // only): each stage's dequantised B^T serves two M = 256 MMA blocks, which
  // halves the dequantisation per MMA; the two accumulators fill the 512 TMEM
  // columns, so they are single-buffered (the epilogue of a tile does not
  // overlap the next tile's MMAs).
  static constexpr int kMBlocks = MB;
  static constexpr int kRowsPerTile = 256 * MB;
  static constexpr int kAccBufs = 2 / MB;
  static constexpr int kASlotBytes = MB * kABytes;
  // Epilogue chunk: EC fp32 columns of a warp's 32 rows per TMEM load and per
  // TMA store (EC = 16: 64-byte rows, 64-byte swizzle; 32: 128-byte rows,
  // 128-byte swizzle; fewer, larger chunks cost less per column).
  static constexpr int kEpiCols = EC;
  static constexpr int kEpiBufBytes = 32 * EC * 4;
  static constexpr int kRawStages = RS;
  static constexpr int kOpStages = OS;
  static constexpr int kAStages = RA;
  static constexpr int kGoBytes = GOB;
  static constexpr int kRawBytes = GOB + kNf4Bytes + kScaleBytes;
  static constexpr int kScaleOff = GOB + kNf4Bytes;  // within a raw slot
  static constexpr int kOpSlotBytes = kPreA ? kBBytes : kOpBytes;
  static constexpr int kBInOp = kPreA ? 0 : kABytes;  // offset of B^T in an operand slot
  static constexpr int kRawOff = 0;
  static constexpr int kAOff = kRawOff + RS * kRawBytes;
  static constexpr int kOpOff = kAOff + RA * MB * kABytes;
  static constexpr int kEpiOff = kOpOff + OS * kOpSlotBytes;
  // Two M-blocks stage every tile's epilogue in the A ring (kEpiInARing), so
  // they need no staging buffers of their own.
  static constexpr int kEpiStageBytes = MB == 2 ? 0 : kEpiWarps * kEpiBufs * kEpiBufBytes;
  static constexpr int kBarOff = kEpiOff + kEpiStageBytes;
  // ... + one barrier per epilogue warp for reading other pairs' partial sums
  static constexpr int kNumBars = 2 * RS + 2 * OS + 2 + 2 + 1 + 2 * RA + kEpiWarps;
  // misc: TMEM address, abort flag, the ready counter (and spare words), then the
  // 16-byte signal words: in CTA 0 one destination per (operand slot,
  // converter warp of a group), and one source.
  static constexpr int kMiscOff = (kBarOff + kNumBars * 8 + 15) & ~15;
  static constexpr int kReadyOff = kMiscOff + 8;
  // Two M-blocks: how many epilogue warps have handed their A-ring staging back
  // (kEpiWarps per item, counted up in item order).
  static constexpr int kRelOff = kMiscOff + 28;
  static constexpr int kSigOff = kMiscOff + 32;
  static constexpr uint32_t kSigSrcOff = kSigOff + OS * kGroupWarps * kSigBytes;
  static constexpr int kSmemBytes = kSigSrcOff + kSigBytes + 1024;  // + alignment slack
  // The pre-converted variant adds one warp: the A-operand producer.
  static constexpr int kThreads = (kWatchWarp + 1 + (kPreA ? 1 : 0)) * 32;  // 736 or 768
  static constexpr int kBoxes = kPreA ? 2 : 4;  // raw-ring boxes per stage
  static_assert(kSmemBytes <= 232448, "shared memory budget");
  static_assert(kRawBytes % 1024 == 0 && kOpSlotBytes % 1024 == 0 && kABytes % 1024 == 0, "align");
  static_assert(kSigOff % 16 == 0 && kSigSrcOff % 16 == 0, "bulk-copy addresses are 16-byte aligned");
  // A pair's last item stages each epilogue warp's M-block (and a finishing
  // pair loads partial sums) in the idle rings: 32 KB per warp.
  static_assert(kEpiWarps * (BK / EC) * kEpiBufBytes <= kEpiOff - kRawOff,
                "the rings hold every epilogue warp's M-block");
  // Two M-blocks: every tile's epilogue stages in the A ring (see kEpiInARing).
  static constexpr bool kEpiInARing = MB == 2;
  static_assert(!kEpiInARing || kEpiWarps * (BK / EC) * kEpiBufBytes <= RA * MB * kABytes,
                "the A ring holds every epilogue warp's M-block");
  // A whole (unsplit) tile's epilogue stages in two A slots, a ring of 16 KB
  // (eight 2 KB chunk buffers) per epilogue warp, two warps per slot, so that
  // the other two slots take the next item's first stages meanwhile.
  static constexpr int kHalfStageBytes = (BK / EC / 2) * kEpiBufBytes;
  static_assert(!kEpiInARing || (RA == 4 && kEpiWarps == 4 && 2 * kHalfStageBytes == MB * kABytes),
                "two epilogue warps' half M-blocks fill one A slot");
  static_assert(kReadyOff + 4 * OS <= kRelOff && kRelOff + 4 <= kSigOff,
                "ready and release counters fit before the signal area");
  static_assert(RS * kBoxes <= 32 && RA <= 32, "one producer lane per (ring slot, box)");
  // Each raw slot must always be consumed by the same converter group.  A group
  // waits for a slot's phase by parity only; if the slot alternated between the
  // groups, a group could wait for phase k while phase k-1 (the other group's
  // stage, copy still in flight) is incomplete, and the completed phase k-2 has
  // the same parity: the wait would pass on stale data.  The same holds for the
  // operand slots, whose release the groups also wait for by parity.
  static_assert(RS % kConvGroups == 0 && OS % kConvGroups == 0,
                "ring slots are not shared between converter groups");
  static_assert(MB == 1 || (MB == 2 && kPreA), "two M-blocks only with the pre-converted A");
};
using LayoutF32 = Layout<2, 4, 2 * kGoBoxBytes>;  // any fp32 grad_out in the launch
using LayoutBF16 = Layout<2, 4, kGoBoxBytes>;     // bf16 grad_out only
using LayoutPreA = Layout<6, 4, 0, 6, 32>;        // grad_out pre-converted to f16
using LayoutPreA2 = Layout<4, 4, 0, 4, 16, 2>;    // pre-converted, 512-token pair tiles

// B^T operand (MN-major, 128-byte swizzle): 64 output columns k per swizzle row,
// 8 rows n per 1024-byte atom; atoms along k are kBLbo apart, atoms along n 1 KB.
constexpr uint32_t kBLbo = BN * 128;  // 8 KB: all 8 n-groups of one 64-k chunk
constexpr uint32_t kSbo = 1024;

// ------------------------------------------------------------------ problems
struct ProblemDesc {  // 128-byte aligned (CUtensorMap); copied as 16-byte words
  CUtensorMap tm_go;      // grad_out [M][N], box 128 rows x 128 bytes, 128B swizzle
  CUtensorMap tm_nf4;     // codes [N][K/2] bytes, box 64 rows x 64 bytes, 64B swizzle
  CUtensorMap tm_out;     // grad_A [M][K] fp32, box 32 rows x 16 columns, 64B swizzle
  CUtensorMap tm_scales;  // scales [N][K/64] fp32, box 64 rows x 4 (if scale_tma)
  const float* scales;
  float* grad_A;
  int M, N, K, dtype;
  int tiles_m, tiles_k, n_stages, tile_begin;  // tiles_m counts 256-row pair tiles
  // 1: the block scales of a stage travel with its NF4 bytes as one more TMA
  // box (needs K % 256 == 0 and 16-byte aligned scales, so that the scale rows
  // are 16-byte strided); 0: each converter thread loads its scale from global
  // memory a turn ahead of its use.
  int scale_tma;
  // 1: the forward product C[M x N] = A[M x K] @ dequant(B_nf4[K x N]) (the
  // shared dimension is K): tm_go holds A (f16), tm_nf4 boxes are 128 rows n x
  // 32 bytes (one 64-k block per row, no swizzle), tm_out is C, M/N/K keep
  // their forward meaning, tiles_k counts 256-column tiles of N and n_stages
  // the 64-wide stages of K.  Pre-converted variant only; scale_tma is 0.
  int fwd;
  // Streamed grouped launch (SkArgs::streamed): per 256-row block of the A
  // operand, the count of slabs (slab_rows rows each) the concurrent f16 pass
  // has finished writing; the A producer waits for a block's full count before
  // its first copy from it.  nullptr otherwise.
  const unsigned int* ready;
  // Pass jobs counted into each ready word: the parts of a fused problem write
  // their column slices of the same rows (1 for a plain problem).
  int ready_parts;
  // Rows of one pass slab of this problem (8, 16, 32 or 64: divides 256).
  int slab_rows;
  // Tile order: 1 = output-column tiles fastest over all row blocks; G > 1 =
  // groups of G row blocks, column tiles slowest within a group, so that the
  // pairs running at the same time share both a few row blocks of A and a few
  // column blocks of the weight in L2.
  int row_group;
};

static_assert(sizeof(ProblemDesc) % 16 == 0, "descriptor copy granularity");
static_assert(sizeof(ProblemDesc) == 640, "descriptor size (the no-allocation array holds 256)");

// One pair tile of one problem, with the problem's fields read once into
// registers (the inline-asm memory clobbers would otherwise force reloads).
struct Tile {
  const ProblemDesc* p;
  const float* scales;
  int M, N, K, dtype;
  int mt, kt, ns, stma, fwd;
};

__device__ __forceinline__ Tile tile_fields(const ProblemDesc& d, const ProblemDesc* p, int t) {
  Tile r;
  r.p = p;
  r.scales = d.scales;
  r.M = d.M;
  r.N = d.N;
  r.K = d.K;
  r.dtype = d.dtype;
  // Output-column tiles vary fastest: the pairs running at the same time then
  // share a few 256-row blocks of grad_out, which stay in L2 while every column
  // tile of them is computed (row-block-fastest order made them stream grad_out
  // from DRAM once per column tile when it does not fit in L2).
  const int local = t - d.tile_begin;
  const int tk = d.tiles_k;
  const int G = d.row_group;
  if (G > 1) {
    const int per_group = G * tk;
    const int g = local / per_group;
    const int idx = local - g * per_group;
    const int rows = min(G, d.tiles_m - g * G);  // the last group may be shorter
    r.kt = idx / rows;
    r.mt = g * G + (idx - r.kt * rows);
  } else {
    r.mt = local / tk;
    r.kt = local % tk;
  }
  r.ns = d.n_stages;
  r.stma = d.scale_tma;
  r.fwd = d.fwd;
  return r;
}

// Tile t of the launch: of the single problem passed by value (its fields are
// read from the kernel's parameters, no global-memory round trip before the
// first copies), or of the grouped launch's descriptor array.
__device__ __forceinline__ Tile tile_at(const ProblemDesc& single, const ProblemDesc* batch,
                                        int count, int t) {
  if (batch == nullptr) return tile_fields(single, &single, t);
  int lo = 0, hi = count - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (batch[mid].tile_begin <= t) lo = mid; else hi = mid - 1;
  }
  return tile_fields(batch[lo], batch + lo, t);
}

// Two M-blocks: the A slots (bit i = slot i of RA) in which an item's epilogue
// stages its result, given the global stage count `it_next` at which the next
// item starts.  A part of a split tile stages whole M-blocks (every slot); a
// whole tile goes through a 16 KB chunk ring per warp in the two slots that
// the next item fills third and fourth, so its first two stages load meanwhile.
template <int RA>
__device__ __forceinline__ uint32_t epi_stage_slots(bool split_part, uint32_t it_next) {
  return split_part ? (1u << RA) - 1u
                    : (1u << ((it_next + 2u) % RA)) | (1u << ((it_next + 3u) % RA));
}

// ------------------------------------------------------------------ work schedule
// The work of a launch is a list of pair tiles, each a run of n_stages stages
// (64 columns of the shared dimension N each).  Tiles [0, dp_tiles) go whole to
// the pairs, round-robin.  When a single problem has too few tiles to keep every
// pair busy for a whole number of waves, the remaining tiles [dp_tiles,
// dp_tiles + sk_tiles) are cut by stages instead ("stream-K"): their stages,
// numbered consecutively, are split into one contiguous run per pair.  A tile
// whose stages fall to several pairs is finished by the pair holding its first
// stage, which processes that part last of all its work; the others (later
// stages of the tile, processed first) leave their fp32 partial sums in a
// workspace and count a flag up, and the finishing pair adds them to its own
// sum in pair order before storing the tile.  The split points depend only on
// the problem and the number of pairs, so results are reproducible.
struct SkArgs {
  int dp_tiles;          // tiles done whole (all tiles when sk_tiles == 0)
  int sk_tiles;          // tiles split by stages (single problem only)
  int stages;            // stages per tile of the split region
  float* partials;       // [pair][rank][BM][BK] fp32 partial sums
  unsigned int* flags;   // [pair] epilogue warps (of both CTAs) done writing partials
  // 1: the f16 A operands are written by a pass that runs beside this kernel
  // (to_f16_stream_kernel) and signals each finished row block through the
  // problem's `ready` counters; the kernel then does not wait for the
  // preceding launch to complete (griddepcontrol.wait) but for those counters.
  int streamed;
};

// One piece of a pair's work: stages [s0, s1) of tile t (s1 clipped to the
// tile's stage count by the caller for whole tiles).
struct Item {
  int t, s0, s1;
};

__host__ __device__ __forceinline__ int64_t sk_start(const SkArgs& sk, int q, int pairs) {
  const int64_t W = static_cast<int64_t>(sk.sk_tiles) * sk.stages;
  return W * q / pairs;
}

// Item k of pair c (k = 0, 1, ...); t < 0 when the pair has no more work.
__host__ __device__ __forceinline__ Item item_at(const SkArgs& sk, int c, int pairs, int k) {
  Item w;
  const int ndp = c < sk.dp_tiles ? (sk.dp_tiles - 1 - c) / pairs + 1 : 0;
  if (k < ndp) {
    w.t = c + k * pairs;
    w.s0 = 0;
    w.s1 = INT_MAX;
    return w;
  }
  w.t = -1;
  w.s0 = w.s1 = 0;
  if (sk.sk_tiles == 0) return w;
  const int64_t st = sk_start(sk, c, pairs), en = sk_start(sk, c + 1, pairs);
  const int64_t tile = st / sk.stages + (k - ndp);
  const int64_t base = tile * sk.stages;
  if (st >= en || base >= en) return w;
  w.t = sk.dp_tiles + static_cast<int>(tile);
  w.s0 = static_cast<int>(st > base ? st - base : 0);
  w.s1 = static_cast<int>(en - base < sk.stages ? en - base : sk.stages);
  return w;
}

// Whether pair q holds any split-region stage (with fewer such stages than
// pairs, some pairs hold none; they write no partial sum).
__host__ __device__ __forceinline__ bool sk_has_stages(const SkArgs& sk, int q, int pairs) {
  return sk_start(sk, q, pairs) < sk_start(sk, q + 1, pairs);
}

// The pair that holds split-region stage x.
__host__ __device__ __forceinline__ int sk_owner(const SkArgs& sk, int64_t x, int pairs) {
  const int64_t W = static_cast<int64_t>(sk.sk_tiles) * sk.stages;
  int q = static_cast<int>((x * pairs) / W);
  if (q > pairs - 1) q = pairs - 1;
  while (q > 0 && sk_start(sk, q, pairs) > x) --q;
  while (q + 1 < pairs && sk_start(sk, q + 1, pairs) <= x) ++q;
  return q;
}

// Stage cursor of a converter group: which item and stage it converts next,
// with the fields of that tile's problem needed for the scale loads.
struct ConvCursor {
  int k, t, s, s1, kt, N, KB;
  bool f32, stma, fwd;
  const float* scales;
};

__device__ __forceinline__ void cc_load(ConvCursor& c, const SkArgs& sk, int cluster, int pairs,
                                        const ProblemDesc& single, const ProblemDesc* batch, int count) {
  const Item w = item_at(sk, cluster, pairs, c.k);
  c.t = w.t;
  if (w.t >= 0) {
    const Tile tl = tile_at(single, batch, count, w.t);
    c.s = w.s0;
    c.s1 = w.s1 < tl.ns ? w.s1 : tl.ns;
    c.kt = tl.kt;
    c.N = tl.N;
    c.KB = tl.K >> 6;
    c.f32 = tl.dtype == NF4_F32;
    c.stma = tl.stma != 0;
    c.fwd = tl.fwd != 0;
    c.scales = tl.scales;
  }
}

__device__ __forceinline__ void cc_start(ConvCursor& c, const SkArgs& sk, int cluster, int pairs,
                                         const ProblemDesc& single, const ProblemDesc* batch, int count) {
  c.k = 0;
  c.s = 0;
  c.s1 = 1;
  c.kt = 0;
  c.N = 0;
  c.KB = 0;
  c.f32 = true;
  c.stma = false;
  c.fwd = false;
  c.scales = nullptr;
  cc_load(c, sk, cluster, pairs, single, batch, count);
}

__device__ __forceinline__ void cc_next(ConvCursor& c, const SkArgs& sk, int cluster, int pairs,
                                        const ProblemDesc& single, const ProblemDesc* batch, int count) {
  if (c.t < 0) return;
  if (++c.s >= c.s1) {
    ++c.k;
    cc_load(c, sk, cluster, pairs, single, batch, count);
  }
}

// Scale of column n = (stage row nl) and global K-block kt*4 + 2*rank + j; 0
// outside the weight, so padded columns dequantise to zero.
__device__ __forceinline__ float cc_scale(const ConvCursor& c, uint32_t rank, int j, int nl) {
  const int n = c.s * BN + nl;
  const int b = c.kt * 4 + 2 * static_cast<int>(rank) + j;
  if (n >= c.N || b >= c.KB) return 0.0f;
  return __ldg(c.scales + static_cast<int64_t>(n) * c.KB + b);
}

// Forward orientation: scale of output column n = kt*256 + 128*rank + r and
// K-block s (the stage); 0 outside the weight.
__device__ __forceinline__ float cc_scale_fwd(const ConvCursor& c, uint32_t rank, int r) {
  const int n = c.kt * BK + static_cast<int>(rank) * BKC + r;
  if (n >= c.N || c.s >= c.KB) return 0.0f;
  return __ldg(c.scales + static_cast<int64_t>(n) * c.KB + c.s);
}



// ------------------------------------------------------------------ kernel
// Progress slots (NF4_PROGRESS builds): 0 producer stages issued, 1 MMA stages
// committed, 2 MMA tiles committed, 3 watcher stages published, 4-19 stages
// finished by converter warp 0-15, 20-23 tiles stored by epilogue warp 0-3.
// At most 72 registers a thread (the launch-bounds limit would be 85): the
// CTA's 768 threads then leave 8,192 registers of the SM for a block of the
// streamed f16 pass beside it.
template <class L>
__global__ void __maxnreg__(72)
    bwd_a_kernel(const __grid_constant__ ProblemDesc single, const ProblemDesc* __restrict__ batch,
                 int count, const __grid_constant__ SkArgs sk) {
  constexpr int kRawStages = L::kRawStages;
  constexpr int kOpStages = L::kOpStages;
  constexpr int kGoBytes = L::kGoBytes;
  constexpr int kRawBytes = L::kRawBytes;
  constexpr int kRawOff = L::kRawOff;
  // A-ring depth, 1 (never used) in the variants without an A ring so that the
  // slot arithmetic below stays well defined.
  constexpr int kAStages = L::kPreA ? L::kAStages : 1;
  constexpr int kMBlocks = L::kMBlocks;
  constexpr int kRowsPerTile = L::kRowsPerTile;
  constexpr uint32_t kAccBufs = L::kAccBufs;
  constexpr uint32_t kASlotBytes = L::kASlotBytes;
  constexpr int kAOff = L::kAOff;
  constexpr int kOpOff = L::kOpOff;
  constexpr int kOpSlotBytes = L::kOpSlotBytes;
  constexpr int kEpiOff = L::kEpiOff;
  constexpr int kBarOff = L::kBarOff;
  constexpr int kMiscOff = L::kMiscOff;
  constexpr int kReadyOff = L::kReadyOff;
  constexpr int kSigOff = L::kSigOff;
  constexpr uint32_t kSigSrcOff = L::kSigSrcOff;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // Pointer arithmetic on the shared array keeps the shared address space
  // visible to the compiler, so plain loads and stores below are ld/st.shared.
  // Both CTAs of a pair get the same offsets (the pair MMA relies on that).
  uint8_t* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  const uint32_t sbase = smem_addr(smem);
  const ProblemDesc* descs = batch != nullptr ? batch : &single;
  const uint32_t rank = cluster_ctarank();          // 0 = leader (issues the MMAs)
  const int cluster = static_cast<int>(blockIdx.x >> 1);
  const int nclusters = static_cast<int>(gridDim.x >> 1);

  const uint32_t bar0 = sbase + kBarOff;
  auto full_raw = [&](uint32_t i) { return bar0 + 8u * i; };
  auto empty_raw = [&](uint32_t i) { return bar0 + 8u * (kRawStages + i); };
  auto full_op = [&](uint32_t i) { return bar0 + 8u * (2 * kRawStages + i); };
  auto empty_op = [&](uint32_t i) { return bar0 + 8u * (2 * kRawStages + kOpStages + i); };
  auto tmem_full = [&](uint32_t i) { return bar0 + 8u * (2 * kRawStages + 2 * kOpStages + i); };
  auto tmem_empty = [&](uint32_t i) {
    return bar0 + 8u * (2 * kRawStages + 2 * kOpStages + 2 + i);
  };
  const uint32_t mma_done = bar0 + 8u * (2 * kRawStages + 2 * kOpStages + 4);
  // Pre-converted variant: A ring.  full_a lives in CTA 0 and counts the bytes
  // of both CTAs' A copies; empty_a is signalled by the MMA commit in both.
  auto full_a = [&](uint32_t i) { return bar0 + 8u * (2 * kRawStages + 2 * kOpStages + 5 + i); };
  auto empty_a = [&](uint32_t i) {
    return bar0 + 8u * (2 * kRawStages + 2 * kOpStages + 5 + kAStages + i);
  };
  // Split tiles: epilogue warp w's barrier for bulk loads of partial sums.
  auto part_bar = [&](uint32_t w) {
    return bar0 + 8u * (2 * kRawStages + 2 * kOpStages + 5 + 2 * L::kAStages + w);
  };
  // Two M-blocks: the epilogue warps hand their A-ring staging back after each
  // item by counting this word up (the A producer may be more than one item
  // behind, so a counter, not the phases of a barrier).
  const uint32_t epi_released = sbase + L::kRelOff;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kMiscOff);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kMiscOff + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  NF4_TRACE_INIT;
  if (threadIdx.x == 0) NF4_PROBE(44, 0);
  // Start the first reads of the problem's descriptor (tensor maps and the
  // fields every role reads) now, so that their latency overlaps the set-up
  // below instead of delaying each role's first stage.
  if (count == 1 && threadIdx.x == 32) {
    tma_prefetch_desc(&descs[0].tm_go);
    tma_prefetch_desc(&descs[0].tm_nf4);
    tma_prefetch_desc(&descs[0].tm_out);
    if (descs[0].scale_tma) tma_prefetch_desc(&descs[0].tm_scales);
  }

  if (threadIdx.x == 0) {
    for (int i = 0; i < kRawStages; ++i) {
      mbar_init(full_raw(i), 1);
      mbar_init(empty_raw(i), kGroupWarps);
    }
    for (int i = 0; i < kOpStages; ++i) {
      // CTA 0's converters, one of which registers with its arrival the bytes
      // of the completion copies of CTA 1's converters (one 16-byte copy per
      // warp; they may land before or after that arrival: the phase completes
      // only when all arrivals and all bytes are in).
      mbar_init(full_op(i), kGroupWarps);
      mbar_init(empty_op(i), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(tmem_full(i), 1);
      mbar_init(tmem_empty(i), 2 * kEpiWarps);  // epilogues of both CTAs (used in CTA 0)
    }
    mbar_init(mma_done, 1);
    for (int i = 0; i < L::kAStages; ++i) {  // none without an A ring
      mbar_init(full_a(i), 1);  // CTA 0's A producer registers both CTAs' bytes
      mbar_init(empty_a(i), 1);
    }
    for (int i = 0; i < kEpiWarps; ++i) mbar_init(part_bar(i), 1);
    for (int i = 0; i < kOpStages; ++i)
      reinterpret_cast<volatile uint32_t*>(smem + kReadyOff)[i] = 0u;
    *reinterpret_cast<volatile uint32_t*>(smem + L::kRelOff) = 0u;
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc_pair(smem_addr(tmem_slot), kTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  // Barriers of both CTAs are initialised before any remote arrive: every role
  // waits for the peer CTA here, except the raw producer, whose copies complete
  // on this CTA's own barriers; it issues its first stages first.
  cluster_arrive();
  if (warp != kProducerWarp) cluster_wait();
  if (threadIdx.x == 0) NF4_PROBE(39, 0);
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == kProducerWarp) {
    // ---------------------------------------------------------------- TMA producer
    // A thread's bulk-tensor copies are served one after another, so every
    // (ring slot, box) pair has its own lane: lane 4*slot + b issues box b of
    // the stages that use `slot` (b = 0 grad_out columns 0-31 (fp32) or 0-63
    // (bf16) and the stage's byte count, b = 1 fp32 columns 32-63, b = 2 the
    // NF4 bytes, b = 3 the block scales; the pre-converted variant has only
    // boxes 2 (with the byte count) and 3, lane 2*slot + b - 2).
    // Stages go in order and lane 0 alone waits for a slot (lanes
    // of one warp waiting on different barriers would wake together).  Boxes may
    // land before the byte count is registered: the phase cannot complete while
    // that arrival is pending.
    const int my_slot = lane / L::kBoxes;
    const int box = L::kPreA ? 2 + (lane & 1) : (lane & 3);
    uint32_t it = 0;
    bool ok = true;
    bool peer_ready = false;  // this warp's cluster_wait done
    for (int k = 0; ok; ++k) {
      const Item w = item_at(sk, cluster, nclusters, k);
      if (w.t < 0) break;
      const Tile tl = tile_at(single, batch, count, w.t);
      const int s1 = w.s1 < tl.ns ? w.s1 : tl.ns;
      const bool f32 = tl.dtype == NF4_F32;
      const uint32_t bytes = (L::kPreA ? 0u : (f32 ? 2u * kGoBoxBytes : kGoBoxBytes)) +
                             kNf4Bytes + (tl.stma ? kScaleBytes : 0u);
      const int row0 = tl.mt * BMP + static_cast<int>(rank) * BM;
      const int x_nf4 = tl.kt * (BK / 2) + static_cast<int>(rank) * (BKC / 2);
      const CUtensorMap* map =
          box == 3 ? &tl.p->tm_scales : (box == 2 ? &tl.p->tm_nf4 : &tl.p->tm_go);
      // x of each box: grad_out column, NF4 byte column, or the first of the
      // pair tile's 4 block scales (4 floats = 16 bytes per k-tile).
      const int x_box = box == 3 ? tl.kt * 4 : (box == 2 ? x_nf4 : 32 * box);
      const bool my_box = box == 3 ? tl.stma != 0 : (box != 1 || f32);
      const bool registers = L::kPreA ? box == 2 : box == 0;
      for (int s = w.s0; s < s1; ++s, ++it) {
        if (!peer_ready && it == static_cast<uint32_t>(kRawStages)) {  // the ring's first fill is out
          cluster_wait();
          peer_ready = true;
        }
        const uint32_t slot = it % kRawStages;
        bool free_slot = true;
        if (lane == 0) free_slot = mbar_wait(empty_raw(slot), ((it / kRawStages) & 1u) ^ 1u, abort_flag);
        if (!__shfl_sync(0xFFFFFFFFu, free_slot, 0)) {
          ok = false;
          break;
        }
        if (my_box && my_slot == static_cast<int>(slot)) {
          const uint32_t fb = full_raw(slot);
          const uint32_t dst =
              sbase + kRawOff + slot * kRawBytes +
              (box == 0 ? 0u
                        : (box == 1 ? static_cast<uint32_t>(kGoBoxBytes)
                                    : (box == 2 ? static_cast<uint32_t>(kGoBytes)
                                                : static_cast<uint32_t>(L::kScaleOff))));
          if (registers) {
            mbar_arrive_expect_tx(fb, bytes);
            NF4_PROBE(40, it);
          }
          if (tl.fwd && box == 2)  // 128 rows n of this CTA's columns, the stage's 32 bytes
            tma_load_2d(dst, map, s * (BN / 2), tl.kt * BK + static_cast<int>(rank) * BKC, fb);
          else
            tma_load_2d(dst, map, box >= 2 ? x_box : s * BN + x_box, box >= 2 ? s * BN : row0, fb);
        }
        if (lane == 0) NF4_PROGRESS_SET(0, it + 1);
        __syncwarp();
      }
    }
    if (!peer_ready) cluster_wait();  // no more stages than slots
    if (lane == 0) {
      // Every issued copy must land before the CTA may exit.
      for (uint32_t i = (it > kRawStages ? it - kRawStages : 0u); i < it; ++i)
        mbar_wait(full_raw(i % kRawStages), (i / kRawStages) & 1u, nullptr);
      // So must every commit the leader multicasts into this CTA's operand-slot
      // barriers (nobody else waits for the last ones): wait for the last phase
      // of each slot.  Both CTAs run the same stage sequence.
      if (ok) {
        for (uint32_t i = (it > kOpStages ? it - kOpStages : 0u); i < it; ++i)
          mbar_wait_cluster(empty_op(i % kOpStages), (i / kOpStages) & 1u, nullptr);
      }
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    // ---------------------------------------------------------------- MMA issuer (CTA 0)
    if (rank == 0) {
      // The whole warp runs this loop and one elected lane issues the MMAs and
      // commits (a warp-converged issuer keeps their operands in uniform
      // registers, see elect_one).  Per stage: 4 MMAs and the commits; the
      // ready counter is read only when the warp has caught up with it.
      // Descriptors of slot 0 are built once; a slot's are those plus its
      // offset in the 16-byte address field.
      constexpr uint32_t idesc = idesc_f16_f32(2 * BM, BK, /*A K-major*/ 0, /*B MN-major*/ 1);
      const uint64_t a_desc0 = smem_desc_sw128(sbase + (L::kPreA ? kAOff : kOpOff), 16, kSbo);
      const uint64_t b_desc0 = smem_desc_sw128(sbase + kOpOff + L::kBInOp, kBLbo, kSbo);
      constexpr uint32_t kBStep = (2u * kSbo) >> 4;  // +2 n-groups per MMA K-step
      // Forward tiles: B is K-major like A (128 rows n per CTA, 128-byte
      // swizzle), +32 bytes per MMA K-step.
      constexpr uint32_t idesc_fwd = idesc_f16_f32(2 * BM, BK, 0, /*B K-major*/ 0);
      const uint64_t b_desc0_fwd = smem_desc_sw128(sbase + kOpOff + L::kBInOp, 16, kSbo);
      const uint32_t ready0 = sbase + kReadyOff;
      uint32_t it = 0, lt = 0, slot = 0, aslot = 0;
      uint32_t avail = 0;  // stages the watcher has published as ready
      bool ok = true;
      for (int k = 0; ok; ++k, ++lt) {
        const Item w = item_at(sk, cluster, nclusters, k);
        if (w.t < 0) break;
        const Tile tl = tile_at(single, batch, count, w.t);
        const int s1 = w.s1 < tl.ns ? w.s1 : tl.ns;
        const uint32_t acc = lt % kAccBufs;
        const uint32_t id = tl.fwd ? idesc_fwd : idesc;
        const uint64_t bdesc = tl.fwd ? b_desc0_fwd : b_desc0;
        const uint32_t bstep = tl.fwd ? 2u : kBStep;
        if (!__all_sync(0xFFFFFFFFu, mbar_wait_cluster(tmem_empty(acc),
                                                       ((lt / kAccBufs) & 1u) ^ 1u, abort_flag))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * BK;  // M-block b: + b * BK
        for (int s = w.s0; s < s1; ++s) {
          if (lane == 0) NF4_PROBE(32, it);
          // The watcher publishes, in order, how many stages' operand barriers
          // it has seen complete; lane 0 reads the counter again only when the
          // warp has caught up with it, so stages that are already ready go to
          // the tensor core back to back.
          if (avail <= it) {
            uint32_t seen = 0;
            bool got = true;
            if (lane == 0) got = flag_wait_ge(ready0, it + 1u, abort_flag, &seen);
            avail = __shfl_sync(0xFFFFFFFFu, seen, 0);
            if (!__shfl_sync(0xFFFFFFFFu, got, 0)) {
              ok = false;
              break;
            }
          }
          // No tcgen05 fence here: the operands were handed to the async proxy
          // by their writers (fence.proxy.async before the barrier arrive) and
          // lane 0 acquired the barrier's completion through the ready word
          // (shared with the warp by the shuffle); a tcgen05.fence per stage
          // would keep the MMAs of consecutive stages from overlapping.
          if (lane == 0) NF4_PROBE(33, it);
          const uint64_t off = static_cast<uint64_t>((slot * kOpSlotBytes) >> 4);
          const uint64_t a =
              a_desc0 + (L::kPreA ? static_cast<uint64_t>((aslot * kASlotBytes) >> 4) : off);
          const uint64_t b = bdesc + off;
          if (elect_one()) {
            // A: +32 bytes per 16 f16 along the swizzled row; B: +2 n-groups.
#pragma unroll
            for (int mb = 0; mb < kMBlocks; ++mb) {
              const uint32_t dm = d_tmem + static_cast<uint32_t>(mb * BK);
              const uint64_t am = a + static_cast<uint64_t>((mb * kABytes) >> 4);
              tc_mma_f16_pair(dm, am, b, id, s != w.s0 ? 1u : 0u);
              tc_mma_f16_pair(dm, am + 2u, b + bstep, id, 1u);
              tc_mma_f16_pair(dm, am + 4u, b + 2u * bstep, id, 1u);
              tc_mma_f16_pair(dm, am + 6u, b + 3u * bstep, id, 1u);
            }
            tc_commit_pair(empty_op(slot), 0x3);
            if constexpr (L::kPreA) tc_commit_pair(empty_a(aslot), 0x3);
          }
          __syncwarp();
          if (lane == 0) NF4_PROBE(38, it);
          if (lane == 0) NF4_PROGRESS_SET(1, it + 1);
          ++it;
          slot = (slot + 1u == static_cast<uint32_t>(kOpStages)) ? 0u : slot + 1u;
          if constexpr (L::kPreA)
            aslot = (aslot + 1u == static_cast<uint32_t>(kAStages)) ? 0u : aslot + 1u;
        }
        if (!ok) break;
        if (elect_one()) tc_commit_pair(tmem_full(acc), 0x3);
        __syncwarp();
        if (lane == 0) NF4_PROGRESS_SET(2, lt + 1);
      }
      // No MMA may still be writing TMEM (of either CTA) when it is released.
      if (elect_one()) tc_commit_pair(mma_done, 0x1);
      __syncwarp();
      mbar_wait(mma_done, 0, nullptr);
      // The epilogues' arrivals for the last two tiles are not needed by any MMA,
      // but the CTA may not exit while one from the other CTA is still in flight.
      if (ok) {
        for (uint32_t l = (lt > kAccBufs ? lt - kAccBufs : 0u); l < lt; ++l)
          mbar_wait_cluster(tmem_empty(l % kAccBufs), (l / kAccBufs) & 1u, nullptr);
      }
    }
    __syncwarp();
  } else if (warp == kWatchWarp) {
    // ---------------------------------------------------------------- watcher (CTA 0)
    // Absorbs the latency of the operand-barrier waits for the MMA thread: it
    // runs up to kOpStages stages ahead (the converters cannot fill a slot again
    // before its MMAs complete) and publishes each completed stage.
    if (rank == 0 && lane == 0) {
      uint32_t it = 0;
      bool ok = true;
      for (int k = 0; ok; ++k) {
        const Item w = item_at(sk, cluster, nclusters, k);
        if (w.t < 0) break;
        const Tile tl = tile_at(single, batch, count, w.t);
        const int s1 = w.s1 < tl.ns ? w.s1 : tl.ns;
        for (int s = w.s0; s < s1; ++s, ++it) {
          const uint32_t slot = it % kOpStages;
          if constexpr (L::kPreA) {
            if (!mbar_wait_cluster(full_a(it % kAStages), (it / kAStages) & 1u, abort_flag)) {
              ok = false;
              break;
            }
            NF4_PROBE(46, it);
          }
          if (!mbar_wait_cluster(full_op(slot), (it / kOpStages) & 1u, abort_flag)) {
            ok = false;
            break;
          }
          NF4_PROBE(41, it);
          st_release_shared(sbase + kReadyOff, it + 1u);
          NF4_PROGRESS_SET(3, it + 1);
        }
      }
    }
    __syncwarp();
  } else if (L::kPreA && warp == kWatchWarp + 1) {
    // ---------------------------------------------------------------- A producer (pre-converted)
    // Each CTA copies its 128 rows x 64 columns of the f16 grad_out into an A
    // slot as soon as the MMAs that last read the slot are done; both copies
    // complete on CTA 0's full_a barrier, for which CTA 0 registers 2 x 16 KB.
    // Lane `slot` issues the copies of that slot (a thread's bulk copies are
    // served one after another); lane 0 alone waits.
    const uint32_t full_a_leader0 = mapa_shared(full_a(0), 0);
    // The A operand is the pre-pass's output: wait for that kernel (a launch
    // that may overlap it) before the first copy; with a streamed pre-pass,
    // for the row blocks of each tile instead (below).
    if (!sk.streamed) griddep_wait();
    uint32_t it = 0;
    bool ok = true;
    // Two M-blocks: item `held_item`'s epilogue stages its result in the A
    // slots `held` until it counts them back (epi_stage_slots).  A copy into one
    // of them waits for that, and so does the start of the item after next.
    int held_item = -1;
    uint32_t held = 0;
    bool prev_split = false;
    auto wait_released = [&](int j) -> bool {
      bool got = true;
      uint32_t seen = 0;
      if (lane == 0)
        got = flag_wait_ge(epi_released, static_cast<uint32_t>(j + 1) * kEpiWarps, abort_flag, &seen);
      return __shfl_sync(0xFFFFFFFFu, got, 0);
    };
    for (int k = 0; ok; ++k) {
      const Item w = item_at(sk, cluster, nclusters, k);
      if (w.t < 0) break;
      const Tile tl = tile_at(single, batch, count, w.t);
      const int s1 = w.s1 < tl.ns ? w.s1 : tl.ns;
      const int row0 = tl.mt * kRowsPerTile + static_cast<int>(rank) * BM;
      if constexpr (L::kEpiInARing) {
        if (held_item >= 0 && held_item < k - 1) {
          if (!wait_released(held_item)) {
            ok = false;
            break;
          }
          held_item = -1;
        }
        if (k > 0) {
          held_item = k - 1;
          held = epi_stage_slots<kAStages>(prev_split, it);
        }
        prev_split = w.s0 > 0 || s1 < tl.ns;
      }
      const unsigned int* cnt = sk.streamed ? tl.p->ready : nullptr;
      if (cnt != nullptr) {
        // Each M-block of the tile is one 256-row block of A: wait until the
        // pass has written all its slabs (fewer in a last, partial block), then
        // order those generic-proxy writes before the copies.
        // (A problem whose grad_out came in f16 has no pass and no counters.)
        bool ready = true;
        if (lane == 0) {
          for (int b = 0; ready && b < kMBlocks; ++b) {
            const int rb = tl.mt * kMBlocks + b;
            const int rows = tl.M - rb * 256;
            if (rows <= 0) break;
            const int sr = tl.p->slab_rows;
            const unsigned int need = static_cast<unsigned int>(tl.p->ready_parts) *
                                      static_cast<unsigned int>(((rows < 256 ? rows : 256) + sr - 1) / sr);
            ready = flag_wait_global_ge(cnt + rb, need, abort_flag);
          }
          fence_proxy_async_global();
        }
        if (!__shfl_sync(0xFFFFFFFFu, ready, 0)) {
          ok = false;
          break;
        }
      }
      for (int s = w.s0; s < s1; ++s, ++it) {
        const uint32_t slot = it % kAStages;
        if constexpr (L::kEpiInARing) {
          if (held_item >= 0 && ((held >> slot) & 1u) != 0u) {
            if (!wait_released(held_item)) {
              ok = false;
              break;
            }
            held_item = -1;
          }
        }
        bool free_slot = true;
        if (lane == 0)
          free_slot = mbar_wait_cluster(empty_a(slot), ((it / kAStages) & 1u) ^ 1u, abort_flag);
        if (!__shfl_sync(0xFFFFFFFFu, free_slot, 0)) {
          ok = false;
          break;
        }
        // Lane kMBlocks*slot + b issues M-block b's box of the slot.
        if (lane / kMBlocks == static_cast<int>(slot)) {
          const int b = lane % kMBlocks;
          if (rank == 0 && b == 0)
            mbar_arrive_expect_tx(full_a(slot), 2u * kMBlocks * kABytes);
          tma_load_2d_pair(sbase + kAOff + slot * kASlotBytes + b * kABytes, &tl.p->tm_go, s * BN,
                           row0 + b * 256, full_a_leader0 + 8u * slot);
          NF4_PROBE(45, it);
        }
        __syncwarp();
      }
    }
    if (lane == 0 && ok) {
      // The last commits into this CTA's empty_a barriers (they also mean that
      // the last copies landed: their MMAs read them) must arrive before exit.
      for (uint32_t i = (it > kAStages ? it - kAStages : 0u); i < it; ++i)
        mbar_wait_cluster(empty_a(i % kAStages), (i / kAStages) & 1u, nullptr);
    }
    __syncwarp();
  } else if (warp >= kConvWarp0) {
    // ---------------------------------------------------------------- converters
    const int cg_thread = threadIdx.x - kConvWarp0 * 32;  // 0..511
    const int group = cg_thread >> 8;                     // 0..1
    const int ct = cg_thread & 255;                       // thread within the group
    const int ar = ct & (BM - 1);                         // A: row of the CTA's tile
    const int ahalf = ct >> 7;                            // A: 16-byte chunks 4*ahalf .. +3
    const int bn = ct & 63;                               // B: row n of the stage
    const int bj = (ct >> 6) & 1;                         // B: NF4 block of the CTA's half
    const int bh = ct >> 7;                               // B: words 4*bh .. +3 of the block
    const uint32_t aswz = static_cast<uint32_t>(ar & 7);
    const uint32_t bswz = static_cast<uint32_t>(bn & 7);
    const uint32_t qchunk = ((2u * bj + bh) ^ ((static_cast<uint32_t>(bn) >> 1) & 3u)) << 4;
    // Forward orientation: thread (row fr of the CTA's 128 columns n, half fh
    // of the stage's 64 k) -> 16-byte chunks 4*fh .. +3 of the K-major row fr.
    const int fr = ct & (BKC - 1);
    const int fh = ct >> 7;
    // CTA 1: where this warp's stage-completion copy goes in CTA 0.
    const uint32_t gw = static_cast<uint32_t>(ct >> 5);  // warp within the group
    const uint32_t full_op_leader0 = mapa_shared(full_op(0), 0);
    const uint32_t sig_leader0 = mapa_shared(sbase + kSigOff + gw * kSigBytes, 0);

    // `nxt` runs two stages (one group turn) ahead of the stage being converted,
    // so the block scale it needs is loaded a whole turn before its use.
    ConvCursor nxt;
    cc_start(nxt, sk, cluster, nclusters, single, batch, count);
    for (int i = 0; i < group; ++i) cc_next(nxt, sk, cluster, nclusters, single, batch, count);
    // (Scales that travel with the raw stage are read from it instead.)
    bool cur_valid = nxt.t >= 0;
    bool cur_f32 = nxt.f32;
    bool cur_stma = nxt.stma;
    bool cur_fwd = nxt.fwd;
    float scale_cur = !cur_valid || cur_stma ? 0.0f
                      : (cur_fwd ? cc_scale_fwd(nxt, rank, fr) : cc_scale(nxt, rank, bj, bn));
    cc_next(nxt, sk, cluster, nclusters, single, batch, count);
    cc_next(nxt, sk, cluster, nclusters, single, batch, count);
    // This thread's scale within a raw slot's scale box (row bn, 16 bytes per row).
    const uint32_t scale_off = L::kScaleOff + bn * 16 + (2u * rank + bj) * 4u;

    uint32_t it = static_cast<uint32_t>(group);
    while (cur_valid) {
      const float scale_pre = scale_cur;
      const bool f32 = cur_f32;
      const bool stma = cur_stma;
      const bool fwd = cur_fwd;
      cur_valid = nxt.t >= 0;
      cur_f32 = nxt.f32;
      cur_stma = nxt.stma;
      cur_fwd = nxt.fwd;
      scale_cur = !cur_valid || cur_stma ? 0.0f
                  : (cur_fwd ? cc_scale_fwd(nxt, rank, fr) : cc_scale(nxt, rank, bj, bn));
      cc_next(nxt, sk, cluster, nclusters, single, batch, count);
      cc_next(nxt, sk, cluster, nclusters, single, batch, count);

      const uint32_t rslot = it % kRawStages;
      const uint32_t oslot = it % kOpStages;
      const bool probe = (lane == 0);
      const int cw = cg_thread >> 5;  // converter warp 0..15
      if (probe && cw % kGroupWarps == 0) NF4_PROBE(43, it);
      // All lanes wait; the warp goes on only if every lane saw the phase
      // complete, so a timeout never leaves the warp divergent.
      if (!__all_sync(0xFFFFFFFFu, mbar_wait(full_raw(rslot), (it / kRawStages) & 1u, abort_flag)))
        break;
      if (probe && (cg_thread >> 5) % kGroupWarps == 0) NF4_PROBE(42, it);

      // Raw inputs of this thread -> registers; then the raw slot is released.
      const uint8_t* raw = smem + kRawOff + rslot * kRawBytes;
      uint4 g[8];
      if constexpr (L::kPreA) {
        (void)f32;
      } else if (f32) {
        const uint8_t* src = raw + ahalf * kGoBoxBytes + ar * 128;
#pragma unroll
        for (int i = 0; i < 8; ++i)
          g[i] = *reinterpret_cast<const uint4*>(src + ((static_cast<uint32_t>(i) ^ aswz) << 4));
      } else {
        const uint8_t* src = raw + ar * 128;
#pragma unroll
        for (int i = 0; i < 4; ++i)
          g[i] = *reinterpret_cast<const uint4*>(src + (((4u * ahalf + i) ^ aswz) << 4));
      }
      // NF4 bytes: backward, 64-byte swizzled rows n of the tile's 128 k; forward,
      // plain 32-byte rows (one 64-k block) of the CTA's 128 columns n.
      const uint4 q = *reinterpret_cast<const uint4*>(
          raw + kGoBytes + (fwd ? static_cast<uint32_t>(fr * 32 + fh * 16) : bn * (BKC / 2) + qchunk));
      const float scale = stma ? *reinterpret_cast<const float*>(raw + scale_off) : scale_pre;
      // The slot is refilled by TMA (async proxy) once released, so these
      // generic-proxy reads must be ordered before that write by a proxy fence.
      // With at least two raw slots per group the slot is released after the
      // stage's operand writes, so that the one fence there orders both;
      // otherwise here, with a fence of its own, so that the group's next
      // stage does not wait for the refill.
      constexpr bool kLateRawRelease = kRawStages >= 2 * kConvGroups;
      if constexpr (!kLateRawRelease) {
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(empty_raw(rslot));
      }

      if (!__all_sync(0xFFFFFFFFu, mbar_wait_cluster(empty_op(oslot),
                                                     ((it / kOpStages) & 1u) ^ 1u, abort_flag)))
        break;
      if (probe) NF4_PROBE(cw, it);
      uint8_t* a_op = smem + kOpOff + oslot * kOpSlotBytes;
      uint8_t* b_op = a_op + L::kBInOp;

      // grad_out -> f16 A operand (K-major, 128B swizzle: chunk c of row r at c ^ (r % 8)).
      uint8_t* a_row = a_op + ar * 128;
#pragma unroll
      for (int i = 0; i < (L::kPreA ? 0 : 4); ++i) {
        uint4 h;
        if (f32) {
          const uint4 x0 = g[2 * i], x1 = g[2 * i + 1];
          h.x = pack_f16x2(__uint_as_float(x0.x), __uint_as_float(x0.y));
          h.y = pack_f16x2(__uint_as_float(x0.z), __uint_as_float(x0.w));
          h.z = pack_f16x2(__uint_as_float(x1.x), __uint_as_float(x1.y));
          h.w = pack_f16x2(__uint_as_float(x1.z), __uint_as_float(x1.w));
        } else {
          const uint4 w = g[i];
          h.x = pack_f16x2(__uint_as_float(w.x << 16), __uint_as_float(w.x & 0xFFFF0000u));
          h.y = pack_f16x2(__uint_as_float(w.y << 16), __uint_as_float(w.y & 0xFFFF0000u));
          h.z = pack_f16x2(__uint_as_float(w.z << 16), __uint_as_float(w.z & 0xFFFF0000u));
          h.w = pack_f16x2(__uint_as_float(w.w << 16), __uint_as_float(w.w & 0xFFFF0000u));
        }
        *reinterpret_cast<uint4*>(a_row + (((4u * ahalf + i) ^ aswz) << 4)) = h;
      }

      // Half an NF4 block (row n = bn, k = 64*bj + 32*bh .. +31) -> four 16-byte
      // chunks of one 128-byte swizzle row of the MN-major B^T; forward: (row n
      // = fr, k = 32*fh .. +31) -> chunks 4*fh .. +3 of the K-major row fr.
      {
        const BlockTable tb = make_block_table(scale);
        const uint32_t sw = fwd ? static_cast<uint32_t>(fr & 7) : bswz;
        const uint32_t hh = fwd ? static_cast<uint32_t>(fh) : static_cast<uint32_t>(bh);
        uint8_t* dst = b_op + (fwd ? (fr >> 3) * kSbo : bj * kBLbo + (bn >> 3) * kSbo) + sw * 128;
        const uint32_t words[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int e = 0; e < 4; ++e)
          *reinterpret_cast<uint4*>(dst + (((4u * hh + e) ^ sw) << 4)) =
              dequant_word(words[e], tb);
      }
      if (probe) NF4_PROBE(48 + cw, it);
      fence_proxy_async_smem();
      __syncwarp();
      if (probe) NF4_PROBE(64 + cw, it);
      if (lane == 0) {
        if constexpr (kLateRawRelease) mbar_arrive(empty_raw(rslot));
        if (rank == 1) {
          // A 16-byte copy into CTA 0 that completes on CTA 0's operand barrier;
          // issued after this warp's operand writes were handed to the async
          // proxy, never waited for here.
          bulk_copy_to_peer(sig_leader0 + oslot * kGroupWarps * kSigBytes, sbase + kSigSrcOff,
                            kSigBytes, full_op_leader0 + 8u * oslot);
        } else if (gw == 0) {
          mbar_arrive_expect_tx(full_op(oslot), kGroupWarps * kSigBytes);
        } else {
          mbar_arrive(full_op(oslot));
        }
      }
      if (probe) NF4_PROBE(16 + cw, it);
      if (lane == 0) NF4_PROGRESS_SET(4 + cw, it + 1);
      it += kConvGroups;
    }
  } else {
    // ---------------------------------------------------------------- epilogue
    // Per item: a whole tile, or the first stages of a split tile, is read out
    // of TMEM (plus, for a split tile, the other pairs' partial sums in pair
    // order) and stored to grad_A through a staging buffer and TMA stores; the
    // later stages of a split tile are left as a partial sum in this pair's
    // workspace slot, followed by a count-up of the pair's flag.
    const uint32_t tmem_empty_leader0 = mapa_shared(tmem_empty(0), 0);
    // The split flags are zeroed by the preceding pre-pass kernel (a streamed
    // pre-pass runs beside this kernel until its end; there is no split then).
    if constexpr (L::kPreA) {
      if (!sk.streamed) griddep_wait();
    }
    constexpr int kEpiCols = L::kEpiCols;
    constexpr int kEpiBufBytes = L::kEpiBufBytes;
    constexpr int kPieces = kEpiCols / 4;  // 16-byte pieces per staged row
    uint8_t* const buf0 = smem + kEpiOff + warp * kEpiBufs * kEpiBufBytes;
    uint32_t lt = 0;
    uint32_t it_next = 0;  // global stage count at which the next item starts
    for (int k = 0;; ++k, ++lt) {
      const Item w = item_at(sk, cluster, nclusters, k);
      if (w.t < 0) break;
      const Tile tl = tile_at(single, batch, count, w.t);
      const int s1 = w.s1 < tl.ns ? w.s1 : tl.ns;
      const bool partial = w.s0 > 0;                // later stages of a split tile
      const bool finish = !partial && s1 < tl.ns;  // first stages of a split tile
      it_next += static_cast<uint32_t>(s1 - w.s0);
      // The pair's last item: once its accumulator is full every stage has been
      // consumed, so the operand rings are idle and serve as deep staging (a
      // warp's whole M-block of chunks, no wait for a staging buffer).
      // With two M-blocks every item stages in the A ring (epi_stage_slots): a
      // whole tile in two of its slots (a 16 KB chunk ring per warp), a part of
      // a split tile in all of it; the A producer refills those slots only
      // after the epilogue has counted them back.
      const bool deep = L::kEpiInARing || item_at(sk, cluster, nclusters, k + 1).t < 0;
      // Pairs whose partial sums complete this tile: cluster+1 .. q_last.
      int q_last = cluster;
      if (finish) {
        const int64_t x_last = static_cast<int64_t>(w.t - sk.dp_tiles) * sk.stages + sk.stages - 1;
        q_last = sk_owner(sk, x_last, nclusters);
      }
      const uint32_t acc = lt % kAccBufs;
      const bool got = mbar_wait_cluster(tmem_full(acc), (lt / kAccBufs) & 1u, abort_flag);
      if (!__all_sync(0xFFFFFFFFu, got)) break;
      if (threadIdx.x == 0) NF4_PROBE(35, lt);
      tc_fence_after();
      if (finish) {
        // The other pairs wrote their parts first thing; wait for all of them.
        bool ready = true;
        if (lane == 0) {
          for (int q = cluster + 1; ready && q <= q_last; ++q)
            if (sk_has_stages(sk, q, nclusters))
              ready = flag_wait_global_ge(sk.flags + q, 2u * kEpiWarps, abort_flag);
        }
        if (!__shfl_sync(0xFFFFFFFFu, ready, 0)) break;
        if (threadIdx.x == 0) NF4_PROBE(37, k);
      }
      // M-block 0's rows and accumulator (block b: + 256 rows, + b * BK columns).
      const int row0 = tl.mt * kRowsPerTile + static_cast<int>(rank) * BM + warp * 32;
      const uint32_t taddr = tmem_base + acc * BK + (static_cast<uint32_t>(warp * 32) << 16);
      // Partial sums move as this warp's 16 staging-layout chunks (2 KB each,
      // 32 KB per warp) between its slot in the workspace and shared memory.
      constexpr uint32_t kWarpPartBytes = (BK / kEpiCols) * kEpiBufBytes;  // 32 KB
      // Pair q's slot: [q][M-block][rank][epilogue warp] x kWarpPartBytes.
      // This warp's 32 KB of the rings (deep staging; a finishing pair's
      // partial-sum loads): in the A ring with two M-blocks, else from the
      // start of the rings (idle during a pair's last item).
      constexpr int kRegionOff = L::kEpiInARing ? L::kAOff : kRawOff;
      const uint32_t region = sbase + kRegionOff + static_cast<uint32_t>(warp) * kWarpPartBytes;
      uint8_t* const region_ptr = smem + kRegionOff + warp * kWarpPartBytes;
      auto warp_slot = [&](int q, int mb) {
        return reinterpret_cast<uint8_t*>(sk.partials) +
               (((static_cast<size_t>(q) * kMBlocks + mb) * 2 + rank) * kEpiWarps + warp) *
                   kWarpPartBytes;
      };
      // Row `lane` of a 32-row chunk, swizzled as the TMA stores to grad_A
      // read it (16-byte piece q of row r at q ^ ((r / 2) % 4) for 64-byte
      // rows, q ^ (r % 8) for 128-byte rows); the partial sums keep the layout.
      const uint32_t sw = kEpiCols == 16 ? (static_cast<uint32_t>(lane) >> 1) & 3u
                                         : static_cast<uint32_t>(lane) & 7u;
      auto stage_chunk = [&](uint8_t* buf, const uint32_t (&r)[kEpiCols]) {
#pragma unroll
        for (int q4 = 0; q4 < kPieces; ++q4)
          *reinterpret_cast<uint4*>(buf + lane * (kEpiCols * 4) + ((static_cast<uint32_t>(q4) ^ sw) << 4)) =
              make_uint4(r[4 * q4], r[4 * q4 + 1], r[4 * q4 + 2], r[4 * q4 + 3]);
      };
      // One 16-column chunk in r: through a staging buffer to grad_A (TMA
      // store) or, for the later stages of a split tile, to this pair's slot.
      // c: column chunk of the M-block; seq: running chunk count of the item
      // (selects the staging buffer).
      auto emit_chunk = [&](int c, int seq, const uint32_t (&r)[kEpiCols], int mb) {
        // Deep staging: chunk c of the M-block has its own place in the rings.
        // Otherwise two staging buffers: at most one copy may still be
        // reading, so the one that last used this buffer is done with it.
        uint8_t* const buf = deep ? region_ptr + c * kEpiBufBytes : buf0 + (seq & 1) * kEpiBufBytes;
        if (threadIdx.x == 0) NF4_PROBE(80, lt * 16 + c);
        if (!deep && lane == 0) bulk_wait_read<kEpiBufs - 1>();
        __syncwarp();
        if (threadIdx.x == 0) NF4_PROBE(81, lt * 16 + c);
        stage_chunk(buf, r);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          if (partial)
            bulk_store_s2g(warp_slot(cluster, mb) + c * kEpiBufBytes, smem_addr(buf), kEpiBufBytes);
          else
            tma_store_2d(&tl.p->tm_out, tl.kt * BK + c * kEpiCols, row0 + mb * 256, smem_addr(buf));
          bulk_commit();
        }
        if (threadIdx.x == 0) NF4_PROBE(82, lt * 16 + c);
      };
      if (L::kEpiInARing && !finish && !partial) {
        // A whole tile (two M-blocks): this warp's 32 chunks go through a ring
        // of 8 staging buffers, its half of one of the two A slots named by
        // epi_stage_slots (warps 0-1: the first, 2-3: the second).  Two chunks
        // per step: TMEM loads, then (once the stores of the chunks 8 earlier
        // have read these buffers) staging, one proxy fence, two stores of one
        // bulk group each.  TMEM drains as far ahead of the stores as the ring
        // allows and goes back to the MMAs with the last loads.
        constexpr int kChunks = BK / kEpiCols;  // per M-block
        constexpr int kRing = L::kHalfStageBytes / kEpiBufBytes;
        constexpr int kTotal = kMBlocks * kChunks;
        static_assert(kRing % 2 == 0 && kRing >= 4 && kRing <= 9 && kChunks % 2 == 0,
                      "two chunks per step; at most 7 bulk groups left pending");
        const uint32_t hs = (it_next + 2u + static_cast<uint32_t>(warp >> 1)) % kAStages;
        const uint32_t hoff = kAOff + hs * kASlotBytes + static_cast<uint32_t>(warp & 1) * L::kHalfStageBytes;
#pragma unroll 1
        for (int i = 0; i < kTotal; i += 2) {
          const int mb = i / kChunks;
          const int cc = i % kChunks;
          uint32_t r[kEpiCols], r2[kEpiCols];
          tmem_ld_cols<kEpiCols>(taddr + mb * BK + cc * kEpiCols, r);
          tmem_ld_cols<kEpiCols>(taddr + mb * BK + (cc + 1) * kEpiCols, r2);
          tmem_wait_ld();
          if (threadIdx.x == 0) NF4_PROBE(83, i);
          if (i + 2 == kTotal) {
            // Every accumulator column has been read: hand TMEM to the next
            // tile's MMAs before the last stores go out.
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
              if (rank == 0) mbar_arrive(tmem_empty(acc));
              else mbar_arrive_remote(tmem_empty_leader0 + 8u * acc);
            }
          }
          if (i >= kRing) {
            // Chunks i - kRing and i - kRing + 1 used these buffers: their
            // stores are the oldest two of the last kRing bulk groups.
            if (lane == 0) bulk_wait_read<kRing - 2>();
            __syncwarp();
          }
          const uint32_t b0 = hoff + static_cast<uint32_t>(i % kRing) * kEpiBufBytes;
          stage_chunk(smem + b0, r);
          stage_chunk(smem + b0 + kEpiBufBytes, r2);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_2d(&tl.p->tm_out, tl.kt * BK + cc * kEpiCols, row0 + mb * 256, sbase + b0);
            bulk_commit();
            tma_store_2d(&tl.p->tm_out, tl.kt * BK + (cc + 1) * kEpiCols, row0 + mb * 256,
                         sbase + b0 + kEpiBufBytes);
            bulk_commit();
          }
          if (threadIdx.x == 0) NF4_PROBE(82, i);
        }
      } else if (!finish && deep) {
        // The pair's last item: the warp stages its whole M-block in the
        // region (chunk c at c x kEpiBufBytes, the staging layout), then
        // one proxy fence and all of the M-block's stores.
#pragma unroll 1
        for (int mb = 0; mb < kMBlocks; ++mb) {
          if (mb > 0) {  // the previous M-block's stores must have read the region
            if (lane == 0) bulk_wait_read<0>();
            __syncwarp();
          }
#pragma unroll 1
          for (int c = 0; c < BK / kEpiCols; ++c) {
            uint32_t r[kEpiCols];
            tmem_ld_cols<kEpiCols>(taddr + mb * BK + c * kEpiCols, r);
            tmem_wait_ld();
            if (threadIdx.x == 0) NF4_PROBE(83, mb * 16 + c);
            stage_chunk(region_ptr + c * kEpiBufBytes, r);
            if (threadIdx.x == 0) NF4_PROBE(80, mb * 16 + c);
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (threadIdx.x == 0) NF4_PROBE(81, mb);
          if (lane == 0) {
            if (partial) {
              bulk_store_s2g(warp_slot(cluster, mb), region, kWarpPartBytes);
            } else {
#pragma unroll 1
              for (int c = 0; c < BK / kEpiCols; ++c)
                tma_store_2d(&tl.p->tm_out, tl.kt * BK + c * kEpiCols, row0 + mb * 256,
                             region + c * kEpiBufBytes);
            }
            bulk_commit();
          }
          if (threadIdx.x == 0) NF4_PROBE(82, mb);
        }
      } else if (!finish) {
#pragma unroll 1
        for (int mb = 0; mb < kMBlocks; ++mb) {
          if constexpr (kEpiCols == 16) {
            // Two 16-column chunks per TMEM wait: one load latency per pair.
#pragma unroll 1
            for (int c = 0; c < BK / kEpiCols; c += 2) {
              uint32_t r[kEpiCols], r2[kEpiCols];
              if (threadIdx.x == 0) NF4_PROBE(83, lt * 16 + c);
              tmem_ld_cols<kEpiCols>(taddr + mb * BK + c * kEpiCols, r);
              tmem_ld_cols<kEpiCols>(taddr + mb * BK + (c + 1) * kEpiCols, r2);
              tmem_wait_ld();
              emit_chunk(c, mb * (BK / kEpiCols) + c, r, mb);
              emit_chunk(c + 1, mb * (BK / kEpiCols) + c + 1, r2, mb);
            }
          } else {
#pragma unroll 1
            for (int c = 0; c < BK / kEpiCols; ++c) {
              uint32_t r[kEpiCols];
              if (threadIdx.x == 0) NF4_PROBE(83, lt * 16 + c);
              tmem_ld_cols<kEpiCols>(taddr + mb * BK + c * kEpiCols, r);
              tmem_wait_ld();
              emit_chunk(c, mb * (BK / kEpiCols) + c, r, mb);
            }
          }
        }
      } else {
        // First stages of a split tile, this pair's last item: its MMAs are
        // done, so the operand rings are free.  Each contributing pair's
        // partial sums (32 KB for this warp) are bulk-loaded into the rings
        // and added to the accumulator in pair order; the last one goes out
        // with the result, the earlier ones back into TMEM.
        uint32_t j = 0;  // loads so far: the parity of part_bar
        bool ok_load = true;
        for (int mb = 0; ok_load && mb < kMBlocks; ++mb)
        for (int q = cluster + 1; ok_load && q <= q_last; ++q) {
          if (!sk_has_stages(sk, q, nclusters)) continue;
          bool more = false;  // another contributor after q
          for (int q2 = q + 1; q2 <= q_last; ++q2) more = more || sk_has_stages(sk, q2, nclusters);
          if (lane == 0) {
            // Stores of the previous M-block's result (deep staging in this
            // region) must have read it; generic reads of the region (previous
            // contributor) and the acquire of the counts come before the
            // async-proxy copy.
            bulk_wait_read<0>();
            fence_proxy_async_smem();
            fence_proxy_async_global();
            mbar_arrive_expect_tx(part_bar(warp), kWarpPartBytes);
            bulk_load_g2s(region, warp_slot(q, mb), kWarpPartBytes, part_bar(warp));
          }
          ok_load = __all_sync(0xFFFFFFFFu, mbar_wait(part_bar(warp), j & 1u, abort_flag));
          if (!ok_load) break;
#pragma unroll 1
          for (int c = 0; c < BK / kEpiCols; ++c) {
            uint32_t r[kEpiCols];
            tmem_ld_cols<kEpiCols>(taddr + mb * BK + c * kEpiCols, r);
            tmem_wait_ld();
            const uint8_t* src = region_ptr + c * kEpiBufBytes + lane * (kEpiCols * 4);
#pragma unroll
            for (int q4 = 0; q4 < kPieces; ++q4) {
              const float4 v = *reinterpret_cast<const float4*>(src + ((static_cast<uint32_t>(q4) ^ sw) << 4));
              r[4 * q4] = __float_as_uint(__uint_as_float(r[4 * q4]) + v.x);
              r[4 * q4 + 1] = __float_as_uint(__uint_as_float(r[4 * q4 + 1]) + v.y);
              r[4 * q4 + 2] = __float_as_uint(__uint_as_float(r[4 * q4 + 2]) + v.z);
              r[4 * q4 + 3] = __float_as_uint(__uint_as_float(r[4 * q4 + 3]) + v.w);
            }
            if (more) {
              tmem_st_cols<kEpiCols>(taddr + mb * BK + c * kEpiCols, r);
            } else {
              emit_chunk(c, mb * (BK / kEpiCols) + c, r, mb);
            }
          }
          if (more) tmem_wait_st();
          __syncwarp();
          ++j;
        }
        if (!ok_load) break;
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (!(L::kEpiInARing && !finish && !partial)) {  // (that path handed TMEM back already)
          if (rank == 0) mbar_arrive(tmem_empty(acc));
          else mbar_arrive_remote(tmem_empty_leader0 + 8u * acc);
        }
        if constexpr (L::kEpiInARing) {
          bulk_wait_read<0>();  // the stores have read the staged result
          red_release_shared_add(epi_released, 1u);
        }
        if (partial) {
          // The warp's partial sums are in global memory once its copies have
          // completed; then they are made visible to generic-proxy readers and
          // this warp is counted in.
          bulk_wait<0>();
          fence_proxy_async_global();
          __threadfence();
          red_release_gpu_add(sk.flags + cluster, 1u);
        }
      }
      if (partial && threadIdx.x == 0) NF4_PROBE(34, k);
      if (threadIdx.x == 0) NF4_PROBE(36, lt);
      if (lane == 0) NF4_PROGRESS_SET(20 + warp, lt + 1);
    }
    if (lane == 0) bulk_wait<0>();
    __syncwarp();
    if (threadIdx.x == 0) NF4_PROBE(84, 0);
  }

  tc_fence_before();
  if (threadIdx.x == 0) NF4_PROBE(44, 1);
  __syncthreads();
  cluster_sync();  // the leader's MMAs are done and no remote arrive is in flight
  if (threadIdx.x == 0) NF4_PROBE(44, 2);
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, kTmemCols);
  }
  // After a wait gave up, CTA 1's converter warps may still have 16-byte signal
  // copies in flight into this CTA's shared memory (on the normal path the
  // watcher waits for all of them): keep the CTA resident for a bounded time
  // so that they land before its shared memory is released.
  // In the pre-converted variant CTA 1's own A copies complete only on CTA 0's
  // barrier, so CTA 1 cannot see them land: it lingers too.
  if ((rank == 0 || L::kPreA) && threadIdx.x == 0 &&
      (*abort_flag != 0 || *(volatile unsigned int*)&g_status != 0)) {
    const long long t0 = clock64();
    while (clock64() - t0 < kAbortLingerCycles) {
    }
  }
}

}  // namespace nf4
