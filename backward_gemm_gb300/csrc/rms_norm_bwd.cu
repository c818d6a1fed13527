// rms_norm_bwd.cu -- backward of RMS layer normalisation, the step upstream of
// the projections' backward in a transformer layer (page "trueno-gpu 0.4.17 --
// src/kernels/backward/rms_norm.rs", module doc "Mathematical Specification").
//
// Forward, per row of `hidden` elements: y_i = x_i * gamma_i / r with
// r = sqrt(mean(x^2) + eps), r stored by the forward pass.  With g = dL/dy:
//
//     dL/dx_i   = gamma_i * g_i / r - x_i * mean_j(x_j * g_j * gamma_j) / r^3
//     dL/dgamma_i = sum over rows of g_i * x_i / r
//
// This is the gradient of the stated forward, which the page's falsifiable
// prediction (agreement with finite differences) fixes.  The page's printed
// formula and kernel differ from it in two ways, both taken as defects: the
// correction term is multiplied by gamma_i as well, and eps is added to r^2 a
// second time although r already holds it.  The page's kernel also limits the
// row to one warp (hidden <= 32) and leaves out dL/dgamma.
//
// Design (HBM-bound: 12 bytes per element of a row, read x and g, write dL/dx):
// a CTA of T threads takes rows blockIdx.x, + gridDim.x, ..., two at a time
// (both rows' loads in flight together); thread t owns the
// float4 columns t, t + T, ... (V of them at most), keeps gamma for them in
// registers and the rows' dL/dgamma contributions too.  The row's dot product
// is reduced by warp shuffles and a fixed-order sum over the warps, so results
// do not depend on timing; each CTA writes its dL/dgamma partial row to the
// workspace and a second kernel sums the partial rows column by column in CTA
// order.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>

#include "nf4_common.h"

namespace nf4 {
namespace rmsb {

constexpr int kMaxWarps = 16;

__device__ __forceinline__ float4 ld_stream(const float4* p) {
  float4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ void st_stream(float4* p, float4 v) {
  asm volatile("st.global.cs.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(v.x), "f"(v.y),
               "f"(v.z), "f"(v.w)
               : "memory");
}

template <int T, int V>
__global__ void __launch_bounds__(T) rows_kernel(const float4* __restrict__ x,
                                                 const float4* __restrict__ gamma,
                                                 const float* __restrict__ rms,
                                                 const float4* __restrict__ gy,
                                                 float4* __restrict__ gx,
                                                 float4* __restrict__ partial, int rows,
                                                 int hidden) {
  constexpr int kWarps = T / 32;
  static_assert(kWarps <= kMaxWarps, "block size");
  // [parity][row of the pair][warp]
  __shared__ float red[2][2][kWarps];
  const int h4 = hidden >> 2;
  const int t = threadIdx.x;
  const int lane = t & 31, warp = t >> 5;
  float4 gam[V], acc[V];
#pragma unroll
  for (int j = 0; j < V; ++j) {
    const int c = t + j * T;
    gam[j] = c < h4 ? __ldg(gamma + c) : make_float4(0.f, 0.f, 0.f, 0.f);
    acc[j] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  const float inv_h = 1.0f / static_cast<float>(hidden);
  const int G = gridDim.x;
  int parity = 0;
  // Two of the CTA's rows per turn (blockIdx.x + 2*i*G and + G): both rows'
  // loads are in flight together, and one barrier serves both reductions.
  for (int row0 = blockIdx.x; row0 < rows; row0 += 2 * G, parity ^= 1) {
    const bool two = row0 + G < rows;
    float4 xv[2][V], gv[2][V];
    float dot[2] = {0.0f, 0.0f};
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const int64_t base = static_cast<int64_t>(row0 + q * G) * h4;
#pragma unroll
      for (int j = 0; j < V; ++j) {
        const int c = t + j * T;
        if (c < h4 && (q == 0 || two)) {
          xv[q][j] = ld_stream(x + base + c);
          gv[q][j] = ld_stream(gy + base + c);
        } else {
          xv[q][j] = make_float4(0.f, 0.f, 0.f, 0.f);
          gv[q][j] = xv[q][j];
        }
      }
    }
#pragma unroll
    for (int q = 0; q < 2; ++q) {
#pragma unroll
      for (int j = 0; j < V; ++j) {
        dot[q] += xv[q][j].x * gv[q][j].x * gam[j].x;
        dot[q] += xv[q][j].y * gv[q][j].y * gam[j].y;
        dot[q] += xv[q][j].z * gv[q][j].z * gam[j].z;
        dot[q] += xv[q][j].w * gv[q][j].w * gam[j].w;
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) dot[q] += __shfl_xor_sync(0xFFFFFFFFu, dot[q], o);
    }
    // Two reduction slots alternate by turn, so one barrier per turn suffices:
    // a slot is rewritten two turns later, after the next turn's barrier.
    if (lane == 0) {
      red[parity][0][warp] = dot[0];
      red[parity][1][warp] = dot[1];
    }
    __syncthreads();
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      if (q == 1 && !two) break;
      const int64_t base = static_cast<int64_t>(row0 + q * G) * h4;
      float total = 0.0f;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) total += red[parity][q][w];
      const float inv_r = 1.0f / __ldg(rms + row0 + q * G);
      // mean(x g gamma) / r^2: the factor of x_i in the correction term.
      const float corr = total * inv_h * inv_r * inv_r;
#pragma unroll
      for (int j = 0; j < V; ++j) {
        const int c = t + j * T;
        if (c < h4) {
          float4 o;
          o.x = inv_r * (gam[j].x * gv[q][j].x - xv[q][j].x * corr);
          o.y = inv_r * (gam[j].y * gv[q][j].y - xv[q][j].y * corr);
          o.z = inv_r * (gam[j].z * gv[q][j].z - xv[q][j].z * corr);
          o.w = inv_r * (gam[j].w * gv[q][j].w - xv[q][j].w * corr);
          st_stream(gx + base + c, o);
          acc[j].x += gv[q][j].x * xv[q][j].x * inv_r;
          acc[j].y += gv[q][j].y * xv[q][j].y * inv_r;
          acc[j].z += gv[q][j].z * xv[q][j].z * inv_r;
          acc[j].w += gv[q][j].w * xv[q][j].w * inv_r;
        }
      }
    }
  }
  if (partial != nullptr) {
    float4* prow = partial + static_cast<int64_t>(blockIdx.x) * h4;
#pragma unroll
    for (int j = 0; j < V; ++j) {
      const int c = t + j * T;
      if (c < h4) prow[c] = acc[j];
    }
  }
}

// dL/dgamma_i = the sum of the CTAs' partial rows.  A CTA takes 32 columns;
// warp w of its kGammaWarps sums the partial rows w, w + kGammaWarps, ... in
// order (lane = column, so each load is one coalesced 128-byte row piece; up
// to 8 of them in flight per warp), then the warp sums are added in warp
// order: a fixed order, so the result does not depend on timing.  The partial
// rows are few (4 per SM) and the sum is latency bound, so it is spread over
// many warps.
constexpr int kGammaWarps = 32;

__global__ void __launch_bounds__(kGammaWarps * 32)
    gamma_kernel(const float* __restrict__ partial, int parts, int hidden,
                 float* __restrict__ dgamma) {
  __shared__ float sums[kGammaWarps][32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int i = blockIdx.x * 32 + lane;
  float s = 0.0f;
  if (i < hidden) {
#pragma unroll 8
    for (int b = warp; b < parts; b += kGammaWarps) s += partial[static_cast<int64_t>(b) * hidden + i];
  }
  sums[warp][lane] = s;
  __syncthreads();
  if (warp == 0 && i < hidden) {
    float total = 0.0f;
#pragma unroll
    for (int w = 0; w < kGammaWarps; ++w) total += sums[w][lane];
    dgamma[i] = total;
  }
}

struct Plan {
  int threads, per;  // block size and float4 columns per thread
};

// Smallest block (128, 256 or 512 threads) whose threads cover the row with at
// most 4 float4 columns each (hidden <= 8192: x, g, gamma and the dL/dgamma
// sums of 4 columns stay in registers).
inline Plan plan_for(int hidden) {
  const int h4 = hidden / 4;
  if (h4 <= 128) return {128, 1};
  if (h4 <= 256) return {128, 2};
  if (h4 <= 512) return {128, 4};
  if (h4 <= 1024) return {256, 4};
  return {512, 4};
}

// CTAs of a launch: 4 per SM (two rows in flight each) when dL/dgamma is
// wanted -- each CTA then writes a partial row, so more CTAs cost partial-sum
// traffic -- and 8 per SM otherwise.
inline int grid_for(int rows, bool with_gamma) {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
    sms = 1;
  return std::max(1, std::min(rows, (with_gamma ? 4 : 8) * sms));
}

}  // namespace rmsb
}  // namespace nf4

using namespace nf4;

extern "C" size_t rms_norm_backward_ws_bytes(int num_rows, int hidden_dim) {
  if (num_rows <= 0 || hidden_dim <= 0) return 0;
  return sizeof(float) * static_cast<size_t>(rmsb::grid_for(num_rows, true)) *
         static_cast<size_t>(hidden_dim);
}

extern "C" int rms_norm_backward(const float* input, const float* gamma, const float* rms,
                                 const float* grad_output, float* grad_input, float* grad_gamma,
                                 int num_rows, int hidden_dim, void* workspace,
                                 size_t workspace_bytes, void* stream) {
  if (num_rows < 0 || hidden_dim <= 0 || hidden_dim % 4 != 0 || hidden_dim > 8192)
    return NF4_ERR_INVALID;
  if (num_rows == 0) {
    if (grad_gamma == nullptr) return NF4_OK;
    return cudaMemsetAsync(grad_gamma, 0, sizeof(float) * hidden_dim, as_stream(stream)) ==
                   cudaSuccess
               ? NF4_OK
               : NF4_ERR_CUDA;
  }
  if (!input || !gamma || !rms || !grad_output || !grad_input) return NF4_ERR_INVALID;
  if (!aligned(input, 16) || !aligned(gamma, 16) || !aligned(grad_output, 16) ||
      !aligned(grad_input, 16) || !aligned(rms, 4) || (grad_gamma && !aligned(grad_gamma, 4)))
    return NF4_ERR_ALIGN;
  const int grid = rmsb::grid_for(num_rows, grad_gamma != nullptr);
  float* partial = nullptr;
  if (grad_gamma != nullptr) {
    if (workspace == nullptr || !aligned(workspace, 16) ||
        workspace_bytes < sizeof(float) * static_cast<size_t>(grid) * hidden_dim)
      return NF4_ERR_WORKSPACE;
    partial = static_cast<float*>(workspace);
  }
  const rmsb::Plan pl = rmsb::plan_for(hidden_dim);
  const cudaStream_t st = as_stream(stream);
  const auto* x4 = reinterpret_cast<const float4*>(input);
  const auto* g4 = reinterpret_cast<const float4*>(gamma);
  const auto* y4 = reinterpret_cast<const float4*>(grad_output);
  auto* o4 = reinterpret_cast<float4*>(grad_input);
  auto* p4 = reinterpret_cast<float4*>(partial);
#define NF4_RMSB_LAUNCH(T, V)                                                                 \
  rmsb::rows_kernel<T, V><<<grid, T, 0, st>>>(x4, g4, rms, y4, o4, p4, num_rows, hidden_dim)
  if (pl.threads == 128 && pl.per == 1) NF4_RMSB_LAUNCH(128, 1);
  else if (pl.threads == 128 && pl.per == 2) NF4_RMSB_LAUNCH(128, 2);
  else if (pl.threads == 128) NF4_RMSB_LAUNCH(128, 4);
  else if (pl.threads == 256) NF4_RMSB_LAUNCH(256, 4);
  else NF4_RMSB_LAUNCH(512, 4);
#undef NF4_RMSB_LAUNCH
  if (cudaGetLastError() != cudaSuccess) return NF4_ERR_CUDA;
  if (grad_gamma != nullptr) {
    rmsb::gamma_kernel<<<(hidden_dim + 31) / 32, rmsb::kGammaWarps * 32, 0, st>>>(
        partial, grid, hidden_dim, grad_gamma);
    if (cudaGetLastError() != cudaSuccess) return NF4_ERR_CUDA;
  }
  return NF4_OK;
}
