// small_m_host.cuh -- host side of the few-token kernel (nf4_small_m.cuh):
// descriptor, cluster-size choice from the device's cluster occupancy, launch.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "host_plan.cuh"
#include "nf4_small_m.cuh"

namespace nf4 {

// ------------------------------------------------------------------ small M
namespace small_m {

static std::atomic<int> g_max_m{64};

static int fill(SmallDesc* d, const void* go, int dtype, const float* scales, const uint8_t* data,
                float* grad_A, int M, int N, int K, int mp) {
  std::memset(d, 0, sizeof(*d));
  const bool f32 = dtype == NF4_F32;
  if (!encode_2d(&d->tm_go, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                 go, static_cast<uint64_t>(N), static_cast<uint64_t>(M),
                 static_cast<uint64_t>(N) * (f32 ? 4 : 2), f32 ? 32 : 64, static_cast<uint32_t>(mp),
                 CU_TENSOR_MAP_SWIZZLE_128B))
    return NF4_ERR_CUDA;
  if (!encode_2d(&d->tm_nf4, CU_TENSOR_MAP_DATA_TYPE_UINT8, data, static_cast<uint64_t>(K / 2),
                 static_cast<uint64_t>(N), static_cast<uint64_t>(K / 2), SK / 2, SN,
                 CU_TENSOR_MAP_SWIZZLE_128B))
    return NF4_ERR_CUDA;
  const int KB = K / 64;
  d->scale_tma = 0;
  if (KB % 4 == 0 && aligned(scales, 16)) {
    if (!encode_2d(&d->tm_scales, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, scales,
                   static_cast<uint64_t>(KB), static_cast<uint64_t>(N),
                   static_cast<uint64_t>(KB) * 4, SK / 64, SN, CU_TENSOR_MAP_SWIZZLE_NONE))
      return NF4_ERR_CUDA;
    d->scale_tma = 1;
  }
  d->scales = scales;
  d->grad_A = grad_A;
  d->M = M;
  d->N = N;
  d->K = K;
  d->dtype = dtype;
  return NF4_OK;
}

// Clusters of S CTAs of configuration C that fit on the current device at once,
// for every S = 1..kMaxCluster (0 where S does not fit), and the SM count.
template <class C>
static int occupancy(const int** clusters, int* sms_out) {
  static int cached[64][kMaxCluster + 1];
  static int sms_cached[64];
  static bool done[64];
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return NF4_ERR_CUDA;
  std::lock_guard<std::mutex> lock(mu);
  if (!done[dev]) {
    auto kern = small_m_kernel<C>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes) !=
            cudaSuccess ||
        cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) !=
            cudaSuccess)
      return NF4_ERR_CUDA;
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return NF4_ERR_CUDA;
    for (int S = 1; S <= kMaxCluster; ++S) {
      cudaLaunchConfig_t cfg = {};
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = static_cast<unsigned>(S);
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.gridDim = dim3(static_cast<unsigned>(S * 64), 1, 1);
      cfg.blockDim = dim3(kThreads, 1, 1);
      cfg.dynamicSmemBytes = C::kSmemBytes;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      int n = 0;
      if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
        (void)cudaGetLastError();  // a size the device cannot schedule: not a sticky error
        n = 0;
      }
      cached[dev][S] = n;
    }
    sms_cached[dev] = sms;
    done[dev] = true;
  }
  *clusters = cached[dev];
  *sms_out = sms_cached[dev];
  return NF4_OK;
}

// Cluster size for T k-tiles of `chunks` stages each: the S whose launch keeps
// the most loaded SM busiest for the shortest time, counting the stages of the
// CTAs that share an SM (and whole extra waves if the clusters do not all fit),
// plus a fixed cost per CTA for its start-up and the reduction, worth about 8
// stages: measured on GB300 at M = 16, N = 4096, K = 14336 (56 k-tiles of 64
// stages), S = 1/2/3/4/5/8/16 took 46.9/28.5/39.3/33.4/31.0/45.3/70.5 us; a
// cost of 2 stages had picked S = 5.
static int choose_split(int T, int chunks, const int* clusters, int sms, int* per_out) {
  constexpr int64_t kFixedStages = 8;
  int64_t best = INT64_MAX;
  int best_s = 1, best_per = chunks;
  for (int S = 1; S <= std::min(kMaxCluster, chunks); ++S) {
    const int per = (chunks + S - 1) / S;
    if ((chunks + per - 1) / per != S) continue;  // same slices as a smaller S
    const int64_t fit = clusters[S];
    if (fit <= 0) continue;
    const int64_t live = std::min<int64_t>(T, fit);
    const int64_t waves = (T + fit - 1) / fit;
    const int64_t per_sm = (live * S + sms - 1) / sms;
    const int64_t cost = waves * per_sm * (per + kFixedStages);
    if (cost < best) {
      best = cost;
      best_s = S;
      best_per = per;
    }
  }
  *per_out = best_per;
  return best_s;
}

template <class C>
static int launch(SmallDesc& d, cudaStream_t stream) {
  const int* clusters = nullptr;
  int sms = 0;
  int rc = occupancy<C>(&clusters, &sms);
  if (rc != NF4_OK) return rc;
  const int T = (d.K + SK - 1) / SK;
  const int chunks = (d.N + SN - 1) / SN;
  int per = chunks;
  const int S = choose_split(T, chunks, clusters, sms, &per);
  if (clusters[S] <= 0) return NF4_ERR_CUDA;
  d.n_per_cta = per * SN;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(S);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(static_cast<unsigned>(T * S), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, small_m_kernel<C>, d) != cudaSuccess) return NF4_ERR_CUDA;
  return launch_status();
}

static int run(const void* go, int dtype, const float* scales, const uint8_t* data,
               float* grad_A, int M, int N, int K, cudaStream_t stream) {
  const int mp = M <= 16 ? 16 : (M <= 32 ? 32 : 64);
  SmallDesc d;
  const int rc = fill(&d, go, dtype, scales, data, grad_A, M, N, K, mp);
  if (rc != NF4_OK) return rc;
  if (mp == 16) return launch<Cfg16>(d, stream);
  if (mp == 32) return launch<Cfg32>(d, stream);
  return launch<Cfg64>(d, stream);
}

}  // namespace small_m

}  // namespace nf4
