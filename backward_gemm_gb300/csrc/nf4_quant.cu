// nf4_quant.cu -- NF4 quantisation of a dense weight, and the f16 dequantisation
// used to check the GEMM's operand values bit for bit.
//
// Layout (page "aprender-gpu 0.32.0 -- src/kernels/backward/nf4_tensor_core.rs",
// build_ptx "PHASE 2"): scales [N][K/64]; codes of column n contiguous in K,
// element (k, n) in nibble k%2 of byte n*(K/2) + k/2, low nibble = even k.
//
// Both kernels give one thread a (column n, K-block b) pair; a warp covers 32
// consecutive columns of one block, so the reads of the row-major dense weight
// (B[k][n], stride N) are coalesced across the warp.
#include <cuda_runtime.h>

#include <cstdint>

#include "nf4_common.h"
#include "nf4_dequant.cuh"

namespace nf4 {

constexpr int kQuantThreads = 128;

// Nearest codebook entry to y: differences in f32, ties to the lower code.
__device__ __forceinline__ uint32_t nearest_code(float y) {
  uint32_t best = 0;
  float best_d = fabsf(__fsub_rn(y, codebook(0)));
#pragma unroll
  for (int c = 1; c < 16; ++c) {
    const float d = fabsf(__fsub_rn(y, codebook(c)));
    if (d < best_d) {
      best_d = d;
      best = static_cast<uint32_t>(c);
    }
  }
  return best;
}

__global__ void __launch_bounds__(kQuantThreads)
    quantize_kernel(const float* __restrict__ B, int K, int N, uint8_t* __restrict__ data,
                    float* __restrict__ scales) {
  const int n = blockIdx.x * kQuantThreads + threadIdx.x;
  const int b = blockIdx.y;
  if (n >= N) return;
  const int KB = K / 64;
  const float* col = B + static_cast<int64_t>(b) * 64 * N + n;

  float v[64];
  float s = 0.0f;
#pragma unroll
  for (int e = 0; e < 64; ++e) {
    v[e] = __ldg(col + static_cast<int64_t>(e) * N);
    s = fmaxf(s, fabsf(v[e]));
  }
  uint32_t w[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    uint32_t word = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const uint32_t c = (s == 0.0f) ? 7u : nearest_code(__fdiv_rn(v[8 * i + j], s));
      word |= c << (4 * j);
    }
    w[i] = word;
  }
  uint4* dst = reinterpret_cast<uint4*>(data + static_cast<int64_t>(n) * (K / 2) + b * 32);
  dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
  dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
  scales[static_cast<int64_t>(n) * KB + b] = s;
}

__global__ void __launch_bounds__(kQuantThreads)
    dequantize_f16_kernel(const float* __restrict__ scales, const uint8_t* __restrict__ data,
                          int K, int N, uint16_t* __restrict__ bt) {
  const int n = blockIdx.x * kQuantThreads + threadIdx.x;
  const int b = blockIdx.y;
  if (n >= N) return;
  const int KB = K / 64;
  const uint4* src = reinterpret_cast<const uint4*>(data + static_cast<int64_t>(n) * (K / 2) + b * 32);
  const uint4 q0 = __ldg(src);
  const uint4 q1 = __ldg(src + 1);
  const BlockTable t = make_block_table(__ldg(scales + static_cast<int64_t>(n) * KB + b));
  const uint32_t words[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
  uint4* dst = reinterpret_cast<uint4*>(bt + static_cast<int64_t>(n) * K + b * 64);
#pragma unroll
  for (int i = 0; i < 8; ++i) dst[i] = dequant_word(words[i], t);
}

}  // namespace nf4

using namespace nf4;

extern "C" int nf4_quantize(const float* B, int K, int N, uint8_t* data, float* scales,
                            void* stream) {
  if (B == nullptr || data == nullptr || scales == nullptr) return NF4_ERR_INVALID;
  if (K <= 0 || N <= 0 || K % 64 != 0) return NF4_ERR_INVALID;
  if (!aligned(B, 4) || !aligned(data, 16) || !aligned(scales, 4)) return NF4_ERR_ALIGN;
  const dim3 grid((N + kQuantThreads - 1) / kQuantThreads, K / 64);
  quantize_kernel<<<grid, kQuantThreads, 0, as_stream(stream)>>>(B, K, N, data, scales);
  return launch_status();
}

extern "C" int nf4_dequantize_f16(const float* scales, const uint8_t* data, int K, int N,
                                  uint16_t* bt, void* stream) {
  const int rc = check_weight(scales, data, K, N);
  if (rc != NF4_OK) return rc;
  if (bt == nullptr || N <= 0) return NF4_ERR_INVALID;
  if (!aligned(bt, 16)) return NF4_ERR_ALIGN;
  const dim3 grid((N + kQuantThreads - 1) / kQuantThreads, K / 64);
  dequantize_f16_kernel<<<grid, kQuantThreads, 0, as_stream(stream)>>>(scales, data, K, N, bt);
  return launch_status();
}
