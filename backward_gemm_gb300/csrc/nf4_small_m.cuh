// nf4_small_m.cuh -- backward-A for few tokens (M <= 64): the same product,
//
//     grad_A[M x K] = grad_out[M x N] @ dequant(B_nf4[K x N])^T
//
// (page "aprender-gpu 0.32.0 -- src/kernels/backward/nf4_tensor_core.rs",
// struct doc comment and build_ptx phases 1-4).  With M this small the weight
// is streamed once and every element of it is dequantised once: the work is the
// NF4 stream, the dequantisation and the tensor core's reads of the dequantised
// operand, not the arithmetic.  A tcgen05 MMA of M = 128 rows costs the same
// time for any N up to 128 and is at its full rate only at N = 256, so the
// dequantised weight is the N side (256 output columns k per MMA) and grad_out
// the M side (MP real token rows, the others zero).
//
// A tile of 256 output columns is too little work for one SM, so the shared
// dimension N is split over a cluster of S CTAs (S <= 16): CTA r of the
// cluster accumulates the n-slice r of the tile in its tensor memory, and the S
// partial tiles are summed through distributed shared memory in the fixed order
// r = 0..S-1, so the result does not depend on timing.
//
//   CTA         MP tokens (MP in {16, 32, 64}, rows >= M are TMA zero fill) x 256
//               output columns k, over the n-slice of its cluster rank, 64 n per
//               stage (4 MMAs of M = 128, N = 256, K = 16; only A rows < MP are
//               stored: the MMA's rows >= MP read the start of the slot's B
//               operand, and their accumulator rows are never read)
//   warps 0, 18 TMA producers of the even and odd stages.  The copies one
//               thread issues are served one after another, so every (ring slot,
//               box) pair has its own lane: grad_out (one or two boxes of MP rows
//               x 128 bytes) and the NF4 box (64 rows n x 128 bytes = the tile's
//               256 k) of every ring slot are in flight at once.  Two warps on
//               different SM sub-partitions keep the issue rate up next to the
//               busy converter warps
//   warp 1      allocates the TMEM accumulator; one thread issues the MMAs
//   warps 2-17  converters, two groups of 8 warps taking alternate stages:
//               thread (n, j) of a group dequantises NF4 block j (64 k) of row n
//               into the MN-major B operand; grad_out -> f16 K-major A operand.
//               After the last stage the converter warps that own TMEM lanes
//               < MP read the accumulator (tcgen05.ld) into shared memory
//   all warps   reduce: CTA r sums its share of the tile's float4s over the S
//               CTAs' partials (ld.shared::cluster) and stores them to grad_A
#pragma once

namespace nf4 {
namespace small_m {

constexpr int SK = 256;       // output columns k per CTA tile (MMA N)
constexpr int SN = 64;        // shared-dimension slice per stage (4 x MMA K = 16)
constexpr int kMmaM = 128;    // MMA M: token rows of the A operand
constexpr int kProducerWarp = 0;
constexpr int kMmaWarp = 1;
constexpr int kConvWarp0 = 2;
constexpr int kConvGroups = 2;   // group g converts the stages s with s % 2 == g
constexpr int kGroupWarps = 8;   // one thread per (row n, 64-k NF4 block) of a stage
constexpr int kConvWarps = kConvGroups * kGroupWarps;
constexpr int kProducer2Warp = kConvWarp0 + kConvWarps;   // 18
constexpr int kThreads = (kProducer2Warp + 1) * 32;       // 608
constexpr int kNf4Bytes = SN * (SK / 2);                  // 64 rows n x 128 bytes
constexpr int kABytes = kMmaM * SN * 2;                   // 16 KB: what an MMA's A reads
constexpr int kBBytes = SK * SN * 2;                      // 32 KB: 256 k x 64 n, MN-major
constexpr uint32_t kBLbo = SN * 128;                      // 8 KB: one 64-k chunk of B
constexpr uint32_t kSbo = 1024;
constexpr int kScaleBytes = SN * 16;                     // 64 rows n x the tile's 4 block scales
constexpr int kBoxLanes = 4;     // producer lanes per ring slot: grad_out x2, NF4, scales
constexpr int kMaxCluster = 16;
constexpr uint32_t kTmemCols = SK;
constexpr int kPartStride = SK + 4;  // floats per partial-tile row (the pad spreads banks)

template <int MP, int RS, int OS>
struct Config {
  static constexpr int kMp = MP;
  static constexpr int kRawStages = RS;
  static constexpr int kOpStages = OS;
  // Raw stage: grad_out (two 32-column fp32 boxes, or one 64-column bf16 box,
  // MP rows of 128 bytes each, 128-byte swizzle), then the NF4 bytes, then the
  // stage's block scales (when they travel by TMA).
  static constexpr int kGoBoxBytes = MP * 128;
  static constexpr int kGoBytes = 2 * kGoBoxBytes;
  static constexpr int kScaleOff = kGoBytes + kNf4Bytes;
  static constexpr int kRawBytes = kGoBytes + kNf4Bytes + kScaleBytes;
  // Operand slot: the MP real rows of the K-major A operand (128 bytes each),
  // then B.  The MMA reads 128 A rows (16 KB); rows >= MP fall on B's first
  // bytes, which is harmless: accumulator rows >= MP are never read.
  static constexpr int kAReal = MP * 128;
  static constexpr int kOpBytes = kAReal + kBBytes;
  static constexpr int kRawOff = 0;
  static constexpr int kOpOff = RS * kRawBytes;
  static constexpr int kBarOff = kOpOff + OS * kOpBytes;
  static constexpr int kNumBars = 2 * RS + 2 * OS + 1;
  static constexpr int kMiscOff = (kBarOff + kNumBars * 8 + 15) & ~15;
  static constexpr int kSmemBytes = kMiscOff + 16 + 1024;  // + alignment slack
  // The partial tile (fp32 [MP][kPartStride]) reuses the raw ring once the main
  // loop is done.
  static constexpr int kPartialBytes = MP * kPartStride * 4;
  static_assert(kPartialBytes <= RS * kRawBytes, "partial tile fits in the raw ring");
  static_assert(kRawBytes % 1024 == 0 && kOpBytes % 1024 == 0 && kGoBytes % 1024 == 0 &&
                    kAReal % 1024 == 0,
                "stage alignment");
  static_assert(kABytes <= kOpBytes, "an MMA's A reads stay inside the slot");
  static_assert(kSmemBytes <= 232448, "shared memory budget");
  static_assert((RS / 2) * kBoxLanes <= 32, "one producer lane per (slot, box)");
  // Each raw slot must always be consumed by the same converter group: a group
  // waits for a slot's phase by parity only, and a slot shared with the other
  // group could show a completed phase of the same parity two phases back.
  static_assert(RS % kConvGroups == 0, "raw slots are not shared between converter groups");
};

// Operand slots outnumber the converter groups, so that a group can fill its
// next slot while the tensor core still reads the previous one.  The weight
// stream is latency-bound (an NF4 box takes ~2-2.5 us from HBM), so the raw
// ring is as deep as shared memory allows: bytes in flight per SM set the rate.
using Cfg16 = Config<16, 6, 4>;
using Cfg32 = Config<32, 4, 4>;
using Cfg64 = Config<64, 4, 3>;

struct SmallDesc {  // 64-byte aligned (CUtensorMap)
  CUtensorMap tm_go;      // grad_out [M][N], box (32 fp32 | 64 bf16) columns x MP rows, 128B swizzle
  CUtensorMap tm_nf4;     // codes [N][K/2] bytes, box 128 bytes x 64 rows, 128B swizzle
  CUtensorMap tm_scales;  // scales [N][K/64] fp32, box 4 x 64 rows (if scale_tma)
  const float* scales;
  float* grad_A;
  int M, N, K, dtype;
  int n_per_cta;       // n-slice of one cluster rank, a multiple of SN
  // 1: each stage's 64 rows x 4 block scales come as one more TMA box of the
  // raw stage (K % 256 == 0 and 16-byte aligned scales); 0: each converter
  // thread loads its scale from global memory well ahead of its use.
  int scale_tma;
};

__device__ __forceinline__ uint32_t cluster_id_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}

__device__ __forceinline__ float4 ld_cluster_f4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}

// Scale of row n (global) and K-block b; 0 outside the weight, so padded rows
// and columns dequantise to zero.
__device__ __forceinline__ float block_scale(const SmallDesc& d, int n, int b) {
  const int KB = d.K >> 6;
  if (n >= d.N || b >= KB) return 0.0f;
  return __ldg(d.scales + static_cast<int64_t>(n) * KB + b);
}

template <class C>
__global__ void __launch_bounds__(kThreads, 1) small_m_kernel(const __grid_constant__ SmallDesc d) {
  constexpr int MP = C::kMp;
  constexpr int RS = C::kRawStages;
  constexpr int OS = C::kOpStages;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  const uint32_t sbase = smem_addr(smem);

  const uint32_t rank = cluster_ctarank();           // n-slice of this CTA
  const int nclus = static_cast<int>(cluster_nctarank());
  const int kt = static_cast<int>(cluster_id_x());  // k-tile of this cluster
  const int n_begin = static_cast<int>(rank) * d.n_per_cta;
  const int n_end = min(d.N, n_begin + d.n_per_cta);
  const int ns = n_end > n_begin ? (n_end - n_begin + SN - 1) / SN : 0;
  const bool f32 = d.dtype == NF4_F32;

  const uint32_t bar0 = sbase + C::kBarOff;
  auto full_raw = [&](uint32_t i) { return bar0 + 8u * i; };
  auto empty_raw = [&](uint32_t i) { return bar0 + 8u * (RS + i); };
  auto full_op = [&](uint32_t i) { return bar0 + 8u * (2 * RS + i); };
  auto empty_op = [&](uint32_t i) { return bar0 + 8u * (2 * RS + OS + i); };
  const uint32_t acc_full = bar0 + 8u * (2 * RS + 2 * OS);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kMiscOff);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kMiscOff + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  NF4_TRACE_INIT;

  if (threadIdx.x == 0) {
    for (int i = 0; i < RS; ++i) {
      mbar_init(full_raw(i), 1);
      mbar_init(empty_raw(i), kGroupWarps);
    }
    for (int i = 0; i < OS; ++i) {
      mbar_init(full_op(i), kGroupWarps);
      mbar_init(empty_op(i), 1);
    }
    mbar_init(acc_full, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_addr(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  if (threadIdx.x == 0) NF4_PROBE(7, 0);

  if (warp == kProducerWarp || warp == kProducer2Warp) {
    // ---------------------------------------------------------------- TMA producers
    // Producer p takes the stages s with s % 2 == p, in order, and so the ring
    // slots p, p + 2, ...; lane 0 alone waits for a stage's slot (lanes of one
    // warp waiting on different barriers would wake together), then the lanes
    // 3*i + b of the slot's index i issue its box b in one instruction: b = 0
    // grad_out columns 0-31 (fp32) or 0-63 (bf16) and the stage's byte count,
    // b = 1 fp32 columns 32-63, b = 2 the NF4 bytes, b = 3 the block scales.
    // Boxes may land before the byte count is registered: the phase cannot
    // complete while that arrival is pending.
    const int p = warp == kProducerWarp ? 0 : 1;
    const int my_slot = p + 2 * (lane / kBoxLanes), box = lane % kBoxLanes;
    const bool my_box = lane < (RS / 2) * kBoxLanes &&
                        (box == 3 ? d.scale_tma != 0 : (box != 1 || f32));
    const CUtensorMap* my_map = box == 3 ? &d.tm_scales : (box == 2 ? &d.tm_nf4 : &d.tm_go);
    const uint32_t my_dst =
        sbase + C::kRawOff + static_cast<uint32_t>(my_slot) * C::kRawBytes +
        (box == 0 ? 0u : (box == 1 ? C::kGoBoxBytes : (box == 2 ? C::kGoBytes : C::kScaleOff)));
    // x of the NF4 box: the tile's 128 bytes; of the scale box: its 4 blocks.
    const int my_x = box == 3 ? kt * (SK / 64) : kt * (SK / 2);
    if (lane == 0) {
      tma_prefetch_desc(&d.tm_go);
      tma_prefetch_desc(&d.tm_nf4);
    }
    const uint32_t bytes = static_cast<uint32_t>((f32 ? 2 : 1) * C::kGoBoxBytes + kNf4Bytes +
                                                 (d.scale_tma ? kScaleBytes : 0));
    int s = p;
    for (; s < ns; s += 2) {
      const uint32_t slot = s % RS;
      bool free_slot = true;
      if (lane == 0) free_slot = mbar_wait(empty_raw(slot), ((s / RS) & 1) ^ 1, abort_flag);
      if (!__shfl_sync(0xFFFFFFFFu, free_slot, 0)) break;
      if (my_box && my_slot == static_cast<int>(slot)) {
        const uint32_t fb = full_raw(slot);
        const int n0 = n_begin + s * SN;
        if (box == 0) mbar_arrive_expect_tx(fb, bytes);
        tma_load_2d(my_dst, my_map, box >= 2 ? my_x : n0 + 32 * box, box >= 2 ? n0 : 0, fb);
        if (box == 2) NF4_PROBE(0, s);
      }
      __syncwarp();
    }
    // Every issued copy must land before the shared memory is reused or the
    // CTA exits: a slot's last phase completes only when all its boxes have.
    if (lane == 0)
      for (int i = s - 2; i >= p && i >= s - RS; i -= 2) mbar_wait(full_raw(i % RS), (i / RS) & 1, nullptr);
    __syncwarp();
  } else if (warp == kMmaWarp) {
    // ---------------------------------------------------------------- MMA issuer
    // The whole warp runs the loop and one elected lane issues (a converged
    // issuer keeps the MMA operands in uniform registers, see elect_one).
    {
      constexpr uint32_t idesc = idesc_f16_f32(kMmaM, SK, /*A K-major*/ 0, /*B MN-major*/ 1);
      const uint64_t a_desc0 = smem_desc_sw128(sbase + C::kOpOff, 16, kSbo);
      const uint64_t b_desc0 = smem_desc_sw128(sbase + C::kOpOff + C::kAReal, kBLbo, kSbo);
      constexpr uint32_t kBStep = (2u * kSbo) >> 4;  // +2 n-groups per MMA K-step
      int s = 0;
      for (; s < ns; ++s) {
        const uint32_t slot = s % OS;
        if (!__all_sync(0xFFFFFFFFu, mbar_wait(full_op(slot), (s / OS) & 1, abort_flag))) break;
        if (lane == 0) NF4_PROBE(5, s);
        // No tcgen05 fence here: the converters handed the operands to the
        // async proxy (fence.proxy.async before their arrive) and this thread
        // acquired the barrier; a fence per stage would keep the MMAs of
        // consecutive stages from overlapping.
        const uint64_t off = static_cast<uint64_t>((slot * C::kOpBytes) >> 4);
        const uint64_t a = a_desc0 + off, b = b_desc0 + off;
        if (elect_one()) {
          // A: +32 bytes along the swizzled 128-byte row; B: +2 n-groups (2 KB).
          tc_mma_f16(tmem_base, a, b, idesc, s != 0 ? 1u : 0u);
          tc_mma_f16(tmem_base, a + 2u, b + kBStep, idesc, 1u);
          tc_mma_f16(tmem_base, a + 4u, b + 2u * kBStep, idesc, 1u);
          tc_mma_f16(tmem_base, a + 6u, b + 3u * kBStep, idesc, 1u);
          tc_commit(empty_op(slot));
        }
        __syncwarp();
        if (lane == 0) NF4_PROBE(6, s);
      }
      if (s > 0) {
        // Also after giving up: no MMA may still run when TMEM is released.
        if (elect_one()) tc_commit(acc_full);
        __syncwarp();
        mbar_wait(acc_full, 0, nullptr);
        // The commits into the last operand slots are not waited for by anyone
        // else: they must have arrived before the CTA exits.
        if (lane == 0)
          for (int i = (s > OS ? s - OS : 0); i < s; ++i)
            mbar_wait(empty_op(i % OS), (i / OS) & 1, nullptr);
      } else if (lane == 0) {
        mbar_arrive(acc_full);  // nothing was issued (empty slice, or gave up at once)
      }
    }
    __syncwarp();
  } else {
    // ---------------------------------------------------------------- converters
    const int cthread = threadIdx.x - kConvWarp0 * 32;  // 0..511
    const int group = cthread >> 8;
    const int ct = cthread & 255;                  // thread within the group
    const int bn = ct & 63;                        // row n of the stage
    const int bj = ct >> 6;                        // NF4 block (64 k) of the tile
    const uint32_t bswz = static_cast<uint32_t>(bn & 7);
    const uint32_t q_off = C::kGoBytes + bn * (SK / 2);
    constexpr int kGoUnits = MP * 8;               // (row m, 8 n) units of grad_out per stage
    constexpr int kGoIters = (kGoUnits + 255) / 256;

    // Block scales come with the raw stage (scale_tma), or are loaded four
    // group turns (eight stages) before their use.
    const bool stma = d.scale_tma != 0;
    auto scale_of = [&](int st) {
      return !stma && st < ns ? block_scale(d, n_begin + st * SN + bn, kt * (SK / 64) + bj) : 0.0f;
    };
    float sc0 = scale_of(group), sc1 = scale_of(group + kConvGroups);
    float sc2 = scale_of(group + 2 * kConvGroups), sc3 = scale_of(group + 3 * kConvGroups);
    bool ok = true;
    for (int s = group; s < ns; s += kConvGroups) {
      const float scale = sc0;
      sc0 = sc1;
      sc1 = sc2;
      sc2 = sc3;
      sc3 = scale_of(s + 4 * kConvGroups);
      const uint32_t rslot = s % RS;
      const uint32_t oslot = s % OS;
      if (!__all_sync(0xFFFFFFFFu, mbar_wait(full_raw(rslot), (s / RS) & 1, abort_flag))) {
        ok = false;
        break;
      }
      const bool lead = lane == 0 && (ct >> 5) == 0;
      const bool tail = lane == 0 && (ct >> 5) == kGroupWarps - 1;
      if (lead) NF4_PROBE(2, s);
      const uint32_t raw = sbase + C::kRawOff + rslot * C::kRawBytes;
      // NF4 block j of row n: 32 bytes, chunks 2j and 2j+1 of the 128-byte row.
      const uint4 q0 = lds128(raw + q_off + (((2u * bj) ^ bswz) << 4));
      const uint4 q1 = lds128(raw + q_off + (((2u * bj + 1u) ^ bswz) << 4));
      const float scale_v =
          stma ? __uint_as_float(lds32(raw + C::kScaleOff + bn * 16 + bj * 4)) : scale;
      uint4 g[kGoIters][2];
#pragma unroll
      for (int u = 0; u < kGoIters; ++u) {
        const int unit = ct + 256 * u;
        if (unit < kGoUnits) {
          const uint32_t m = static_cast<uint32_t>(unit >> 3), c8 = static_cast<uint32_t>(unit & 7);
          if (f32) {
            // n = 8*c8 .. +7: chunks 2*c8, 2*c8 + 1 (mod 8) of the 32-column box c8 / 4.
            const uint32_t row = raw + (c8 >> 2) * C::kGoBoxBytes + m * 128;
            const uint32_t c0 = (2u * c8) & 7u;
            g[u][0] = lds128(row + ((c0 ^ (m & 7u)) << 4));
            g[u][1] = lds128(row + (((c0 + 1u) ^ (m & 7u)) << 4));
          } else {
            g[u][0] = lds128(raw + m * 128 + ((c8 ^ (m & 7u)) << 4));
          }
        }
      }
      // The raw slot is refilled by TMA (async proxy) once released, so these
      // generic-proxy reads must be ordered before that write: it is released
      // after the stage's operand writes (below), where one proxy fence orders
      // both (every configuration has at least two raw slots per group).
      static_assert(RS >= 2 * kConvGroups, "a group keeps its raw slot through its stage");

      if (!__all_sync(0xFFFFFFFFu, mbar_wait(empty_op(oslot), ((s / OS) & 1) ^ 1, abort_flag))) {
        ok = false;
        break;
      }
      if (lead) NF4_PROBE(3, s);
      const uint32_t a_op = sbase + C::kOpOff + oslot * C::kOpBytes;
      const uint32_t b_op = a_op + C::kAReal;
      // grad_out -> f16 A operand (K-major, 128B swizzle: chunk c8 of row m at c8 ^ (m % 8)).
#pragma unroll
      for (int u = 0; u < kGoIters; ++u) {
        const int unit = ct + 256 * u;
        if (unit < kGoUnits) {
          const uint32_t m = static_cast<uint32_t>(unit >> 3), c8 = static_cast<uint32_t>(unit & 7);
          uint4 hv;
          if (f32) {
            const uint4 x0 = g[u][0], x1 = g[u][1];
            hv.x = pack_f16x2(__uint_as_float(x0.x), __uint_as_float(x0.y));
            hv.y = pack_f16x2(__uint_as_float(x0.z), __uint_as_float(x0.w));
            hv.z = pack_f16x2(__uint_as_float(x1.x), __uint_as_float(x1.y));
            hv.w = pack_f16x2(__uint_as_float(x1.z), __uint_as_float(x1.w));
          } else {
            const uint4 w = g[u][0];
            hv.x = pack_f16x2(__uint_as_float(w.x << 16), __uint_as_float(w.x & 0xFFFF0000u));
            hv.y = pack_f16x2(__uint_as_float(w.y << 16), __uint_as_float(w.y & 0xFFFF0000u));
            hv.z = pack_f16x2(__uint_as_float(w.z << 16), __uint_as_float(w.z & 0xFFFF0000u));
            hv.w = pack_f16x2(__uint_as_float(w.w << 16), __uint_as_float(w.w & 0xFFFF0000u));
          }
          sts128(a_op + m * 128 + ((c8 ^ (m & 7u)) << 4), hv);
        }
      }
      // One NF4 block (row n = bn, k = 64*bj .. +63) -> one 128-byte swizzle row
      // of the MN-major B operand.
      {
        const BlockTable tb = make_block_table(scale_v);
        const uint32_t dst = b_op + bj * kBLbo + (bn >> 3) * kSbo + bswz * 128;
        const uint32_t words[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
#pragma unroll
        for (int e = 0; e < 8; ++e)
          sts128(dst + ((static_cast<uint32_t>(e) ^ bswz) << 4), dequant_word(words[e], tb));
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(empty_raw(rslot));
        mbar_arrive(full_op(oslot));
      }
      if (lead) NF4_PROBE(4, s);
      if (tail) NF4_PROBE(8, s);
    }

    // ---------------------------------------------------------------- accumulator -> partial
    // Converter warp w owns TMEM lanes 32*(w % 4) .. +31, the token rows m; the
    // four warps of each quarter with rows < MP read 64 of the 256 columns k
    // each into the partial tile P[m][k] at the start of the raw ring (every
    // copy into the ring has landed and been read by then).
    const uint32_t quarter = static_cast<uint32_t>(warp & 3);
    if (static_cast<int>(quarter) * 32 < MP) {
      const int part_idx = (warp - kConvWarp0) / 4;  // 0..3 within the quarter
      const bool got = ok && __all_sync(0xFFFFFFFFu, mbar_wait(acc_full, 0, abort_flag));
      if (threadIdx.x == 4 * 32) NF4_PROBE(7, 1);
      const int m = static_cast<int>(quarter) * 32 + lane;
      const uint32_t prow = sbase + C::kRawOff + static_cast<uint32_t>(m * kPartStride * 4);
      if (got && ns > 0) {
        tc_fence_after();
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          const int c = 2 * part_idx + cc;
          uint32_t r[32];
          tmem_ld_32x32b_x32(tmem_base + ((quarter * 32u) << 16) + static_cast<uint32_t>(c * 32), r);
          tmem_wait_ld();
          if (m < MP) {
#pragma unroll
            for (int i = 0; i < 8; ++i)
              sts128(prow + static_cast<uint32_t>((c * 32 + 4 * i) * 4),
                     make_uint4(r[4 * i], r[4 * i + 1], r[4 * i + 2], r[4 * i + 3]));
          }
        }
      } else if (m < MP) {
#pragma unroll 1
        for (int c = 16 * part_idx; c < 16 * part_idx + 16; ++c)
          sts128(prow + static_cast<uint32_t>(c * 16), make_uint4(0, 0, 0, 0));
      }
    }
    tc_fence_before();
  }

  // ---------------------------------------------------------------- cluster reduction
  if (threadIdx.x == kConvWarp0 * 32) NF4_PROBE(7, 2);
  __syncwarp();
  cluster_sync();  // every CTA's partial tile is in its shared memory
  if (threadIdx.x == 0) NF4_PROBE(7, 3);
  {
    const int S = nclus;
    const int e4 = d.M * (SK / 4);  // float4s of the tile's valid rows
    const int per = (e4 + S - 1) / S;
    const int beg = static_cast<int>(rank) * per;
    const int end = min(e4, beg + per);
    const uint32_t part0 = sbase + C::kRawOff;
    for (int e = beg + static_cast<int>(threadIdx.x); e < end; e += kThreads) {
      const int m = e / (SK / 4);
      const int k4 = e % (SK / 4);
      const int kg = kt * SK + 4 * k4;
      if (kg >= d.K) continue;
      const uint32_t off = part0 + static_cast<uint32_t>((m * kPartStride + 4 * k4) * 4);
      // All S loads first (they are independent), then the sum in rank order.
      float4 v[kMaxCluster];
#pragma unroll
      for (int r = 0; r < kMaxCluster; ++r)
        if (r < S) v[r] = ld_cluster_f4(mapa_shared(off, static_cast<uint32_t>(r)));
      float4 acc = v[0];
#pragma unroll
      for (int r = 1; r < kMaxCluster; ++r) {
        if (r < S) {
          acc.x += v[r].x;
          acc.y += v[r].y;
          acc.z += v[r].z;
          acc.w += v[r].w;
        }
      }
      *reinterpret_cast<float4*>(d.grad_A + static_cast<int64_t>(m) * d.K + kg) = acc;
    }
  }
  if (threadIdx.x == 0) NF4_PROBE(7, 4);
  __syncwarp();
  cluster_sync();  // no CTA leaves while another still reads its partial
  if (threadIdx.x == 0) NF4_PROBE(7, 5);
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

}  // namespace small_m
}  // namespace nf4
