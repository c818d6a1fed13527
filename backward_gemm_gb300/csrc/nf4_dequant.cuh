// nf4_dequant.cuh -- NF4 codebook and the per-block dequantisation used by every
// kernel that turns packed NF4 codes into f16 operands.
//
// The value of element (k, n) is f16_rn( f32( scale[n][k/64] * codebook[code] ) )
// (page "aprender-gpu 0.32.0 -- src/kernels/backward/nf4_tensor_core.rs",
// build_ptx "PHASE 2": f32 multiply of the block scale by the codebook entry,
// then an f32 -> f16 conversion).  The codebook is the NormalFloat4 table of
// Dettmers et al., "QLoRA" (2023).
//
// Instead of a select tree per element, each (column, 64-element block) gets a
// 16-entry f16 table built once (16 multiplies + 8 paired conversions), split
// into a low-byte and a high-byte half; eight codes are then looked up with
// byte permutes (prmt): codes 0-7 and 8-15 are looked up separately and merged
// on bit 3 of each code.  The result is bit-identical to the per-element
// multiply-and-convert, because the table holds exactly those 16 products.
#pragma once

#include <cuda_fp16.h>
#include <cstdint>

#include "ptx.cuh"

namespace nf4 {

// NormalFloat4 codebook, ascending (QLoRA, the NF4 data type).
__device__ __forceinline__ float codebook(int c) {
  constexpr float kTable[16] = {
      -1.0f,
      -0.6961928009986877f,
      -0.5250730514526367f,
      -0.39491748809814453f,
      -0.28444138169288635f,
      -0.18477343022823334f,
      -0.09105003625154495f,
      0.0f,
      0.07958029955625534f,
      0.16093020141124725f,
      0.24611230194568634f,
      0.33791524171829224f,
      0.44070982933044434f,
      0.5626170039176941f,
      0.7229568362236023f,
      1.0f,
  };
  return kTable[c];
}

// Low bytes (lo[q]) and high bytes (hi[q]) of the 16 f16 values of one block:
// lo[q] holds the low bytes of entries 4q..4q+3.
struct BlockTable {
  uint32_t lo[4];
  uint32_t hi[4];
};

__device__ __forceinline__ uint32_t pack_f16x2(float a, float b) {
  const __half2 h = __floats2half2_rn(a, b);  // a -> low half, b -> high half, RNE
  return *reinterpret_cast<const uint32_t*>(&h);
}

__device__ __forceinline__ BlockTable make_block_table(float scale) {
  uint32_t p[8];
#pragma unroll
  for (int i = 0; i < 8; ++i)
    p[i] = pack_f16x2(__fmul_rn(scale, codebook(2 * i)), __fmul_rn(scale, codebook(2 * i + 1)));
  BlockTable t;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    t.lo[q] = prmt(p[2 * q], p[2 * q + 1], 0x6420u);  // low bytes of entries 4q..4q+3
    t.hi[q] = prmt(p[2 * q], p[2 * q + 1], 0x7531u);  // high bytes
  }
  return t;
}

// Eight codes (nibble i of v = element i, low nibble first) -> eight f16 values;
// .x holds elements 0 (low half) and 1, .y 2 and 3, .z 4 and 5, .w 6 and 7.
__device__ __forceinline__ uint4 dequant_word(uint32_t v, const BlockTable& t) {
  const uint32_t s = v & 0x77777777u;  // code & 7: byte index into an 8-entry table
  const uint32_t s_hi = s >> 16;
  const uint32_t x = v << 4;
  // 0xFF in byte i where bit 3 of code i is set (prmt sign-replicate on the byte
  // whose most significant bit is that code bit).
  const uint32_t m_lo = prmt(v, x, 0x9D8Cu);
  const uint32_t m_hi = prmt(v, x, 0xBFAEu);

  const uint32_t lo_l = bitselect(m_lo, prmt(t.lo[2], t.lo[3], s), prmt(t.lo[0], t.lo[1], s));
  const uint32_t hi_l = bitselect(m_lo, prmt(t.hi[2], t.hi[3], s), prmt(t.hi[0], t.hi[1], s));
  const uint32_t lo_h =
      bitselect(m_hi, prmt(t.lo[2], t.lo[3], s_hi), prmt(t.lo[0], t.lo[1], s_hi));
  const uint32_t hi_h =
      bitselect(m_hi, prmt(t.hi[2], t.hi[3], s_hi), prmt(t.hi[0], t.hi[1], s_hi));

  uint4 out;
  out.x = prmt(lo_l, hi_l, 0x5140u);
  out.y = prmt(lo_l, hi_l, 0x7362u);
  out.z = prmt(lo_h, hi_h, 0x5140u);
  out.w = prmt(lo_h, hi_h, 0x7362u);
  return out;
}

}  // namespace nf4
