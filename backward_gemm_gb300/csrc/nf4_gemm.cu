// nf4_gemm.cu -- the C ABI entry points of the NF4-dequant-fused backward-A
// GEMM (include/nf4bwd.h):
//
//     grad_A[M x K] = grad_out[M x N] @ dequant(B_nf4[K x N])^T
//
// (page "aprender-gpu 0.32.0 -- src/kernels/backward/nf4_tensor_core.rs",
// struct doc comment and build_ptx phases 1-4.)  The kernels are in
// pair_kernel.cuh (the persistent tcgen05 pair kernel), nf4_small_m.cuh (the
// few-token kernel) and prepass.cuh (f16 pre-pass, descriptor upload); their
// host-side planning and launch code in host_plan.cuh and small_m_host.cuh.
// Everything is compiled as this one translation unit, so that every kernel
// records a timeout in the same device status word that nf4_check_error reads.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <climits>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <vector>

#include "nf4_common.h"
#include "pair_kernel.cuh"
#include "prepass.cuh"
#include "host_plan.cuh"
#include "small_m_host.cuh"
#include "dense_gemm.cuh"

using namespace nf4;

extern "C" int nf4_abi_version(void) { return 1; }

extern "C" int nf4_set_small_m_max(int m_max) {
  if (m_max < 0) m_max = 0;
  if (m_max > 64) m_max = 64;
  return small_m::g_max_m.exchange(m_max);
}

extern "C" int nf4_small_m_split(int N, int K, int sms, int cta_slots, int* per_out) {
  // Host-only planning rule of the small-M kernel: clusters of S CTAs are
  // assumed to fit cta_slots / S times at once.
  if (N <= 0 || K <= 0 || sms <= 0 || cta_slots <= 0 || per_out == nullptr) return -1;
  int fit[small_m::kMaxCluster + 1] = {0};
  for (int S = 1; S <= small_m::kMaxCluster; ++S) fit[S] = cta_slots / S;
  const int T = (K + small_m::SK - 1) / small_m::SK;
  const int chunks = (N + small_m::SN - 1) / small_m::SN;
  return small_m::choose_split(T, chunks, fit, sms, per_out);
}

extern "C" const char* nf4_status_string(int status) {
  switch (status) {
    case NF4_OK: return "ok";
    case NF4_ERR_INVALID: return "invalid argument";
    case NF4_ERR_ALIGN: return "misaligned pointer";
    case NF4_ERR_CUDA: return "CUDA error";
    case NF4_ERR_TIMEOUT: return "kernel wait timed out";
    case NF4_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    default: return "unknown status";
  }
}

extern "C" int nf4_backward_a_ex(const void* grad_out, int go_dtype, const float* scales,
                                 const uint8_t* data, float* grad_A, int M, int N, int K,
                                 void* stream) {
  int rc = check_problem(grad_out, go_dtype, scales, data, grad_A, M, N, K);
  if (rc != NF4_OK || M == 0) return rc;
  if (N == 0) {
    return cudaMemsetAsync(grad_A, 0, sizeof(float) * static_cast<size_t>(M) * K,
                           as_stream(stream)) == cudaSuccess
               ? NF4_OK
               : NF4_ERR_CUDA;
  }
  if (go_dtype == NF4_F16) {
    // Already the A operand's type: the pre-converted kernel reads it as is.
    int pairs = 0;
    rc = max_clusters<LayoutPreA>(&pairs);
    if (rc != NF4_OK) return rc;
    const bool tiles512 = use_tiles512(M, N, K, pairs, /*can_split=*/false);
    ProblemDesc d;
    rc = fill_desc_pre(&d, static_cast<const uint16_t*>(grad_out), scales, data, grad_A, M, N, K,
                       tiles512 ? LayoutPreA2::kRowsPerTile : LayoutPreA::kRowsPerTile);
    if (rc != NF4_OK) return rc;
    const int64_t tiles = static_cast<int64_t>(d.tiles_m) * d.tiles_k;
    if (tiles > INT_MAX) return NF4_ERR_INVALID;
    if (tiles512)
      return launch_layout<LayoutPreA2>(d, nullptr, 1, static_cast<int>(tiles), nullptr,
                                        as_stream(stream));
    return launch_layout<LayoutPreA>(d, nullptr, 1, static_cast<int>(tiles), nullptr,
                                     as_stream(stream));
  }
  if (M <= small_m::g_max_m.load())
    return small_m::run(grad_out, go_dtype, scales, data, grad_A, M, N, K, as_stream(stream));
  ProblemDesc d;
  rc = fill_desc(&d, grad_out, go_dtype, scales, data, grad_A, M, N, K);
  if (rc != NF4_OK) return rc;
  const int64_t tiles = static_cast<int64_t>(d.tiles_m) * d.tiles_k;
  if (tiles > INT_MAX) return NF4_ERR_INVALID;
  return launch(d, nullptr, 1, static_cast<int>(tiles), go_dtype == NF4_BF16, as_stream(stream));
}

extern "C" int nf4_backward_a(const float* grad_out, const float* scales, const uint8_t* data,
                              float* grad_A, int M, int N, int K, void* stream) {
  return nf4_backward_a_ex(grad_out, NF4_F32, scales, data, grad_A, M, N, K, stream);
}


extern "C" int nf4_set_tile_rows(int rows) {
  if (rows != 0 && rows != 256 && rows != 512) return -1;
  return g_tile_rows.exchange(rows);
}

extern "C" int nf4_tile_rows(int M, int N, int K, int pairs, int can_split) {
  if (M <= 0 || N <= 0 || K <= 0 || pairs <= 0) return -1;
  return use_tiles512(M, N, K, pairs, can_split != 0) ? 512 : 256;
}

extern "C" int nf4_split_plan(int tiles, int stages, int pairs, int* dp_tiles, int* sk_tiles) {
  if (tiles <= 0 || stages <= 0 || pairs <= 0 || dp_tiles == nullptr || sk_tiles == nullptr)
    return -1;
  SkArgs sk;
  std::memset(&sk, 0, sizeof(sk));
  plan_split(tiles, stages, pairs, &sk);
  *dp_tiles = sk.dp_tiles;
  *sk_tiles = sk.sk_tiles;
  return 0;
}

extern "C" int nf4_split_item(int tiles, int stages, int pairs, int pair, int k, int* item) {
  if (tiles <= 0 || stages <= 0 || pairs <= 0 || pair < 0 || pair >= pairs || k < 0 ||
      item == nullptr)
    return -1;
  SkArgs sk;
  std::memset(&sk, 0, sizeof(sk));
  plan_split(tiles, stages, pairs, &sk);
  const Item w = item_at(sk, pair, pairs, k);
  if (w.t < 0) return 0;
  item[0] = w.t;
  item[1] = w.s0;
  item[2] = w.s1 < stages ? w.s1 : stages;
  // Pairs whose partial sums the item's epilogue adds (a first-stage item of
  // a split tile): those of item[3] .. item[4] inclusive that hold any stage
  // (nf4_split_item reports them), none when item[4] < item[3].
  item[3] = pair + 1;
  item[4] = pair;
  if (w.t >= sk.dp_tiles && w.s0 == 0 && item[2] < stages)
    item[4] = sk_owner(sk, static_cast<int64_t>(w.t - sk.dp_tiles) * stages + stages - 1, pairs);
  return 1;
}

namespace nf4 {
// One problem on the pre-converted kernel, its descriptor d filled: the split
// plan of a last partial wave (when the workspace holds its flags and partial
// sums), the f16 pre-pass of the A operand a (M rows x R, R the shared
// dimension) into the workspace unless it is f16 already, and the launch.
// With `jobs`, the pre-pass is that grouped pass (the parts of a fused call
// written into their column slices of the workspace's copy) instead of the
// single-source pass over a.
static int launch_pre_single(ProblemDesc& d, const void* a, int a_dtype, int M, int R,
                             void* workspace, size_t workspace_bytes, bool tiles512,
                             cudaStream_t stream, const F16Jobs* jobs = nullptr) {
  const bool f16_in = jobs == nullptr && a_dtype == NF4_F16;
  const int64_t tiles = static_cast<int64_t>(d.tiles_m) * d.tiles_k;
  if (tiles > INT_MAX) return NF4_ERR_INVALID;
  // The split needs its flags and partial sums after the f16 copy; a workspace
  // holding only the copy runs every tile whole.  The plan is made for the
  // number of pairs the chosen kernel runs at once (its launch uses them all).
  int pairs = 0;
  int rc = tiles512 ? max_clusters<LayoutPreA2>(&pairs) : max_clusters<LayoutPreA>(&pairs);
  if (rc != NF4_OK) return rc;
  const size_t base = round256(f16_bytes(M, R));
  SkArgs sk;
  std::memset(&sk, 0, sizeof(sk));
  unsigned int* flags = nullptr;
  int nflags = 0;
  if (workspace_bytes >= base + sk_bytes(pairs)) {
    plan_split(static_cast<int>(tiles), d.n_stages, pairs, &sk);
    if (sk.sk_tiles > 0) {
      uint8_t* w = static_cast<uint8_t*>(workspace) + base;
      flags = reinterpret_cast<unsigned int*>(w);
      nflags = pairs;
      sk.flags = flags;
      sk.partials = reinterpret_cast<float*>(w + round256(sizeof(unsigned int) * pairs));
    }
  }
  if (f16_in || jobs != nullptr) {
    // No single-source pre-pass: zero the split flags on the stream instead.
    if (nflags > 0 &&
        cudaMemsetAsync(flags, 0, sizeof(unsigned int) * nflags, stream) != cudaSuccess)
      return NF4_ERR_CUDA;
    if (jobs != nullptr) {
      rc = launch_f16_jobs(*jobs, stream);
      if (rc != NF4_OK) return rc;
    }
  } else {
    rc = launch_to_f16(a, a_dtype, static_cast<uint16_t*>(workspace), M, R, flags, nflags, stream);
    if (rc != NF4_OK) return rc;
  }
  const SkArgs* skp = sk.sk_tiles > 0 ? &sk : nullptr;
  if (tiles512)
    return launch_layout<LayoutPreA2>(d, nullptr, 1, static_cast<int>(tiles), skp, stream,
                                      /*pdl=*/!f16_in);
  return launch_layout<LayoutPreA>(d, nullptr, 1, static_cast<int>(tiles), skp, stream,
                                   /*pdl=*/!f16_in);
}
}  // namespace nf4

extern "C" size_t nf4_backward_a_ws_bytes(int M, int N) {
  if (M <= 0 || N <= 0) return 0;
  int pairs = 0;
  if (max_clusters<LayoutPreA>(&pairs) != NF4_OK || pairs <= 0) return round256(f16_bytes(M, N));
  return round256(f16_bytes(M, N)) + sk_bytes(pairs);
}

extern "C" int nf4_backward_a_ws(const void* grad_out, int go_dtype, const float* scales,
                                 const uint8_t* data, float* grad_A, int M, int N, int K,
                                 void* workspace, size_t workspace_bytes, void* stream) {
  int rc = check_problem(grad_out, go_dtype, scales, data, grad_A, M, N, K);
  if (rc != NF4_OK || M == 0) return rc;
  if (N == 0) {
    return cudaMemsetAsync(grad_A, 0, sizeof(float) * static_cast<size_t>(M) * K,
                           as_stream(stream)) == cudaSuccess
               ? NF4_OK
               : NF4_ERR_CUDA;
  }
  const bool f16_in = go_dtype == NF4_F16;
  if (!f16_in && M <= small_m::g_max_m.load())
    return small_m::run(grad_out, go_dtype, scales, data, grad_A, M, N, K, as_stream(stream));
  if (workspace == nullptr || !aligned(workspace, 256) || workspace_bytes < f16_bytes(M, N))
    return NF4_ERR_WORKSPACE;
  // f16 grad_out is the A operand already (the copy region goes unused).
  const uint16_t* go_f16 = f16_in ? static_cast<const uint16_t*>(grad_out)
                                  : static_cast<uint16_t*>(workspace);
  int pairs = 0;
  rc = max_clusters<LayoutPreA>(&pairs);
  if (rc != NF4_OK) return rc;
  const bool can_split = workspace_bytes >= round256(f16_bytes(M, N)) + sk_bytes(pairs);
  const bool tiles512 = use_tiles512(M, N, K, pairs, can_split);
  ProblemDesc d;
  rc = fill_desc_pre(&d, go_f16, scales, data, grad_A, M, N, K,
                     tiles512 ? LayoutPreA2::kRowsPerTile : LayoutPreA::kRowsPerTile);
  if (rc != NF4_OK) return rc;
  return launch_pre_single(d, grad_out, go_dtype, M, N, workspace, workspace_bytes, tiles512,
                           as_stream(stream));
}

extern "C" size_t nf4_forward_ws_bytes(int M, int K) { return nf4_backward_a_ws_bytes(M, K); }

extern "C" int nf4_forward_ws(const void* A, int a_dtype, const float* scales, const uint8_t* data,
                              float* C, int M, int N, int K, void* workspace,
                              size_t workspace_bytes, void* stream) {
  if (a_dtype != NF4_F32 && a_dtype != NF4_BF16 && a_dtype != NF4_F16) return NF4_ERR_INVALID;
  if (M < 0 || N < 0 || K <= 0 || K % 64 != 0) return NF4_ERR_INVALID;
  if (M == 0 || N == 0) return NF4_OK;
  if (A == nullptr || scales == nullptr || data == nullptr || C == nullptr) return NF4_ERR_INVALID;
  if (N % 4 != 0) return NF4_ERR_INVALID;  // C rows are 16-byte strided for the TMA stores
  if (!aligned(A, 16) || !aligned(data, 16) || !aligned(scales, 4) || !aligned(C, 16))
    return NF4_ERR_ALIGN;
  const bool f16_in = a_dtype == NF4_F16;
  if (workspace == nullptr || !aligned(workspace, 256) || workspace_bytes < f16_bytes(M, K))
    return NF4_ERR_WORKSPACE;
  const uint16_t* a_f16 = f16_in ? static_cast<const uint16_t*>(A) : static_cast<uint16_t*>(workspace);
  int pairs = 0;
  int rc = max_clusters<LayoutPreA>(&pairs);
  if (rc != NF4_OK) return rc;
  const bool can_split = workspace_bytes >= round256(f16_bytes(M, K)) + sk_bytes(pairs);
  // The shared dimension is K and the output columns are N.
  const bool tiles512 = use_tiles512(M, K, N, pairs, can_split);
  ProblemDesc d;
  rc = fill_desc_fwd(&d, a_f16, scales, data, C, M, N, K,
                     tiles512 ? LayoutPreA2::kRowsPerTile : LayoutPreA::kRowsPerTile);
  if (rc != NF4_OK) return rc;
  return launch_pre_single(d, A, a_dtype, M, K, workspace, workspace_bytes, tiles512,
                           as_stream(stream));
}

extern "C" int nf4_backward_a_fused(const nf4_part* parts, int count, const float* scales,
                                    const uint8_t* data, float* grad_x, int M, int K,
                                    void* workspace, size_t workspace_bytes, void* stream) {
  if (count <= 0 || count > kF16JobsPerLaunch || parts == nullptr) return NF4_ERR_INVALID;
  if (M < 0 || K <= 0 || K % 64 != 0) return NF4_ERR_INVALID;
  int64_t ntot = 0;
  for (int i = 0; i < count; ++i) {
    const nf4_part& p = parts[i];
    if (p.go_dtype != NF4_F32 && p.go_dtype != NF4_BF16 && p.go_dtype != NF4_F16)
      return NF4_ERR_INVALID;
    if (p.N <= 0 || p.N % 8 != 0) return NF4_ERR_INVALID;
    ntot += p.N;
  }
  if (ntot > INT_MAX) return NF4_ERR_INVALID;
  if (M == 0) return NF4_OK;
  if (scales == nullptr || data == nullptr || grad_x == nullptr) return NF4_ERR_INVALID;
  for (int i = 0; i < count; ++i) {
    if (parts[i].grad_out == nullptr) return NF4_ERR_INVALID;
    if (!aligned(parts[i].grad_out, 16)) return NF4_ERR_ALIGN;
  }
  if (!aligned(grad_x, 16) || !aligned(data, 16) || !aligned(scales, 4)) return NF4_ERR_ALIGN;
  const int N = static_cast<int>(ntot);
  if (workspace == nullptr || !aligned(workspace, 256) || workspace_bytes < f16_bytes(M, N))
    return NF4_ERR_WORKSPACE;
  int pairs = 0;
  int rc = max_clusters<LayoutPreA>(&pairs);
  if (rc != NF4_OK) return rc;
  const bool can_split = workspace_bytes >= round256(f16_bytes(M, N)) + sk_bytes(pairs);
  const bool tiles512 = use_tiles512(M, N, K, pairs, can_split);
  uint16_t* a16 = static_cast<uint16_t*>(workspace);
  ProblemDesc d;
  rc = fill_desc_pre(&d, a16, scales, data, grad_x, M, N, K,
                     tiles512 ? LayoutPreA2::kRowsPerTile : LayoutPreA::kRowsPerTile);
  if (rc != NF4_OK) return rc;
  // Part p's grad_out goes into columns [c_p, c_p + N_p) of the f16 A operand
  // (rows N apart; every N_p is a multiple of 8, so every slice starts on a
  // 16-byte boundary and no group of the pass writes into a neighbour's slice).
  F16Jobs jobs;
  std::memset(&jobs, 0, sizeof(jobs));
  jobs.n = count;
  int64_t at = 0;
  int col = 0;
  for (int i = 0; i < count; ++i) {
    const nf4_part& p = parts[i];
    F16Job& j = jobs.job[i];
    j.src = p.grad_out;
    j.dst = a16 + col;
    j.mode = p.go_dtype == NF4_F32 ? kSrcF32 : (p.go_dtype == NF4_BF16 ? kSrcBF16 : kSrcF16);
    j.N = p.N;
    j.ldh = p.N;
    j.pitch = f16_pitch(N);
    j.groups_per_row = (p.N + 15) >> 4;
    j.begin = at;
    at += static_cast<int64_t>(M) * j.groups_per_row;
    col += p.N;
  }
  jobs.end = at;
  return launch_pre_single(d, nullptr, NF4_F16, M, N, workspace, workspace_bytes, tiles512,
                           as_stream(stream), &jobs);
}

extern "C" size_t nf4_backward_a_batched_workspace(int count) {
  if (count <= 0) return 0;
  return sizeof(ProblemDesc) * static_cast<size_t>(count);
}

extern "C" int nf4_backward_a_batched(const nf4_problem* problems, int count, void* workspace,
                                      size_t workspace_bytes, void* stream) {
  if (count < 0 || (count > 0 && problems == nullptr)) return NF4_ERR_INVALID;
  for (int i = 0; i < count; ++i) {
    const nf4_problem& p = problems[i];
    if (p.go_dtype == NF4_F16) return NF4_ERR_INVALID;  // single calls only
    const int rc = check_problem(p.grad_out, p.go_dtype, p.scales, p.data, p.grad_A, p.M, p.N, p.K);
    if (rc != NF4_OK) return rc;
  }
  cudaStream_t st = as_stream(stream);
  std::vector<ProblemDesc> descs;
  descs.reserve(count);
  const int small_max = small_m::g_max_m.load();
  for (int i = 0; i < count; ++i) {
    const nf4_problem& p = problems[i];
    if (p.M == 0) continue;
    if (p.N == 0) {
      if (cudaMemsetAsync(p.grad_A, 0, sizeof(float) * static_cast<size_t>(p.M) * p.K, st) !=
          cudaSuccess)
        return NF4_ERR_CUDA;
      continue;
    }
    if (p.M <= small_max) {
      // Few tokens: the problem's own launch of the few-token kernel, so that
      // it gets the same result as a single call.
      const int rc = small_m::run(p.grad_out, p.go_dtype, p.scales, p.data, p.grad_A, p.M, p.N,
                                  p.K, st);
      if (rc != NF4_OK) return rc;
      continue;
    }
    descs.emplace_back();
    const int rc = fill_desc(&descs.back(), p.grad_out, p.go_dtype, p.scales, p.data, p.grad_A,
                             p.M, p.N, p.K);
    if (rc != NF4_OK) return rc;
  }
  if (descs.empty()) return NF4_OK;
  if (workspace == nullptr || !aligned(workspace, 256) ||
      workspace_bytes < sizeof(ProblemDesc) * descs.size())
    return NF4_ERR_WORKSPACE;
  // Longest tiles first, so that the static round-robin over the flattened
  // tile list ends with the short ones.
  std::stable_sort(descs.begin(), descs.end(), [](const ProblemDesc& a, const ProblemDesc& b) {
    return a.n_stages > b.n_stages;
  });
  int64_t total = 0;
  for (ProblemDesc& d : descs) {
    d.tile_begin = static_cast<int>(total);
    total += static_cast<int64_t>(d.tiles_m) * d.tiles_k;
    if (total > INT_MAX) return NF4_ERR_INVALID;
  }
  ProblemDesc* ws = static_cast<ProblemDesc*>(workspace);
  for (size_t i = 0; i < descs.size(); i += kDescsPerUpload) {
    const int n = static_cast<int>(std::min<size_t>(kDescsPerUpload, descs.size() - i));
    DescChunk chunk;
    std::memset(&chunk, 0, sizeof(chunk));
    std::memcpy(chunk.d, descs.data() + i, sizeof(ProblemDesc) * n);
    upload_descs_kernel<<<1, 256, 0, st>>>(chunk, ws + i, n);
    if (cudaGetLastError() != cudaSuccess) return NF4_ERR_CUDA;
  }
  ProblemDesc unused;
  std::memset(&unused, 0, sizeof(unused));
  bool all_bf16 = true;
  for (const ProblemDesc& d : descs) all_bf16 = all_bf16 && d.dtype == NF4_BF16;
  return launch(unused, static_cast<const ProblemDesc*>(workspace), static_cast<int>(descs.size()),
                static_cast<int>(total), all_bf16, st);
}

// ------------------------------------------------------------------ grouped, pre-converted
namespace nf4 {
// One problem of a grouped pre-converted launch: a plain backward-A problem
// (one part) or a fused one (the parts' grad_out side by side along N, the
// weights stacked along N).
constexpr int kMaxParts = 8;
struct GPart {
  const void* src;
  int dtype, N;
};
struct GProblem {
  GPart part[kMaxParts];
  int nparts;
  const float* scales;
  const uint8_t* data;
  float* out;
  int M, N, K;  // N: the sum of the parts'
};

// A problem that gets an f16 copy: every fused problem, a plain one unless its
// grad_out is f16 already (then it is read in place).
static inline bool needs_copy(const GProblem& p) {
  return p.M > 0 && p.N > 0 && (p.nparts > 1 || p.part[0].dtype != NF4_F16);
}

// A plain problem that the few-token kernel runs on its own.
static inline bool few_token(const GProblem& p, int small_max) {
  return p.nparts == 1 && p.part[0].dtype != NF4_F16 && p.M > 0 && p.N > 0 && p.M <= small_max;
}

static size_t group_copy_bytes(const GProblem* problems, int count) {
  size_t total = 0;
  for (int i = 0; i < count; ++i)
    if (needs_copy(problems[i])) total += round256(f16_bytes(problems[i].M, problems[i].N));
  return total;
}

// Words of the streamed pass's bookkeeping for these problems (0 when the group
// cannot be streamed): the work counter, the per-SM claim flags and one ready
// counter per 256-row block of every problem with a copy.
static size_t stream_words(const GProblem* problems, int count) {
  size_t blocks = 0;
  int jobs = 0;
  for (int i = 0; i < count; ++i) {
    if (!needs_copy(problems[i])) continue;
    jobs += problems[i].nparts;
    blocks += static_cast<size_t>((problems[i].M + 255) / 256);
  }
  if (jobs == 0 || jobs > kStreamMaxJobs) return 0;
  return 1 + kStreamClaimWords + blocks;
}

static size_t grouped_ws_bytes(const GProblem* problems, int count) {
  return round256(sizeof(ProblemDesc) * static_cast<size_t>(count)) +
         group_copy_bytes(problems, count) +
         round256(sizeof(unsigned int) * stream_words(problems, count));
}

// The grouped launch of the pre-converted path over checked problems.
static int grouped_ws(const GProblem* problems, int count, void* workspace, size_t workspace_bytes,
                      cudaStream_t st) {
  const size_t desc_bytes = round256(sizeof(ProblemDesc) * static_cast<size_t>(count));
  // Nothing is enqueued before the workspace is known to be big enough.
  bool any_gemm = false;
  const int small_max = small_m::g_max_m.load();
  for (int i = 0; i < count; ++i) {
    const GProblem& p = problems[i];
    if (p.M > 0 && p.N > 0 && !few_token(p, small_max)) any_gemm = true;
  }
  const size_t copy_bytes = group_copy_bytes(problems, count);
  if (any_gemm && (workspace == nullptr || !aligned(workspace, 256) ||
                   workspace_bytes < desc_bytes + copy_bytes))
    return NF4_ERR_WORKSPACE;
  // Tile size for the whole group: 512 tokens when every GEMM problem has more
  // than 256 tokens, there are at least half a wave of 512-token tiles and the
  // tiles average at least 8 stages (the single-problem rule, on the group).
  int pairs = 0;
  if (any_gemm) {
    const int rc = max_clusters<LayoutPreA>(&pairs);
    if (rc != NF4_OK) return rc;
  }
  int64_t t2 = 0, t2_stages = 0;
  bool all_tall = true;
  for (int i = 0; i < count; ++i) {
    const GProblem& p = problems[i];
    if (p.M == 0 || p.N == 0 || few_token(p, small_max)) continue;
    const int64_t tiles = static_cast<int64_t>((p.M + 511) / 512) * ((p.K + BK - 1) / BK);
    t2 += tiles;
    t2_stages += tiles * ((p.N + BN - 1) / BN);
    all_tall = all_tall && p.M > 256;
  }
  const int forced = g_tile_rows.load();
  const bool tiles512 =
      forced != 0 ? forced == 512
                  : (all_tall && t2 > 0 && tiles512_rule(t2, static_cast<int>(t2_stages / t2), pairs));
  const int rows_per_tile = tiles512 ? LayoutPreA2::kRowsPerTile : LayoutPreA::kRowsPerTile;
  // With room for its bookkeeping after the copies, the f16 pass runs beside
  // the GEMM (to_f16_stream_kernel), otherwise before it.
  const size_t swords = stream_words(problems, count);
  const bool streamed = any_gemm && swords > 0 &&
                        workspace_bytes >= desc_bytes + copy_bytes +
                                               round256(sizeof(unsigned int) * swords);
  unsigned int* stream_area =
      streamed ? reinterpret_cast<unsigned int*>(static_cast<uint8_t*>(workspace) + desc_bytes +
                                                 copy_bytes)
               : nullptr;
  std::vector<ProblemDesc> descs;
  descs.reserve(count);
  std::vector<F16Job> jobs;
  std::vector<int> jobs_of;  // per descriptor: its first f16 job (jobs_n of them), or -1
  std::vector<int> jobs_n;
  uint8_t* copy = static_cast<uint8_t*>(workspace) + desc_bytes;
  for (int i = 0; i < count; ++i) {
    const GProblem& p = problems[i];
    if (p.M == 0) continue;
    if (p.N == 0) {
      if (cudaMemsetAsync(p.out, 0, sizeof(float) * static_cast<size_t>(p.M) * p.K, st) !=
          cudaSuccess)
        return NF4_ERR_CUDA;
      continue;
    }
    uint16_t* dst = nullptr;
    if (needs_copy(p)) {
      dst = reinterpret_cast<uint16_t*>(copy);
      copy += round256(f16_bytes(p.M, p.N));
    }
    if (few_token(p, small_max)) {
      // Few tokens: the problem's own launch of the few-token kernel.
      const int rc = small_m::run(p.part[0].src, p.part[0].dtype, p.scales, p.data, p.out, p.M,
                                  p.N, p.K, st);
      if (rc != NF4_OK) return rc;
      continue;
    }
    descs.emplace_back();
    jobs_of.push_back(dst != nullptr ? static_cast<int>(jobs.size()) : -1);
    jobs_n.push_back(dst != nullptr ? p.nparts : 0);
    const uint16_t* a = dst != nullptr ? dst : static_cast<const uint16_t*>(p.part[0].src);
    const int rc = fill_desc_pre(&descs.back(), a, p.scales, p.data, p.out, p.M, p.N, p.K,
                                 rows_per_tile);
    if (rc != NF4_OK) return rc;
    if (dst != nullptr) {
      // Part j's grad_out goes into its columns of the copy (rows f16_pitch(N)
      // apart; every part of a fused problem is a multiple of 8 columns wide).
      int col = 0;
      for (int q = 0; q < p.nparts; ++q) {
        const GPart& pt = p.part[q];
        F16Job j;
        j.src = pt.src;
        j.dst = dst + col;
        j.mode = pt.dtype == NF4_F32 ? kSrcF32 : (pt.dtype == NF4_BF16 ? kSrcBF16 : kSrcF16);
        j.N = pt.N;
        j.ldh = f16_pitch(pt.N);
        j.pitch = f16_pitch(p.N);
        j.groups_per_row = (j.ldh + 15) >> 4;
        j.begin = static_cast<int64_t>(p.M) * j.groups_per_row;  // size for now
        jobs.push_back(j);
        col += pt.N;
      }
    }
  }
  if (descs.empty()) return NF4_OK;
  // With the pass beside the GEMM, problems with more GEMM work per byte of the
  // pass come first (largest K: the pass writes M x N elements for 2 M N K
  // flops), so that the pass gets ahead while the GEMM works on them; then
  // longest tiles first (stable).
  std::vector<int> order(descs.size());
  for (size_t i = 0; i < order.size(); ++i) order[i] = static_cast<int>(i);
  std::stable_sort(order.begin(), order.end(), [&](int a, int b) {
    if (streamed && descs[a].K != descs[b].K) return descs[a].K > descs[b].K;
    return descs[a].n_stages > descs[b].n_stages;
  });
  {
    std::vector<ProblemDesc> sorted;
    std::vector<int> sorted_of, sorted_n;
    sorted.reserve(descs.size());
    for (int i : order) {
      sorted.push_back(descs[i]);
      sorted_of.push_back(jobs_of[i]);
      sorted_n.push_back(jobs_n[i]);
    }
    descs.swap(sorted);
    jobs_of.swap(sorted_of);
    jobs_n.swap(sorted_n);
  }
  int64_t total = 0;
  for (ProblemDesc& d : descs) {
    d.tile_begin = static_cast<int>(total);
    total += static_cast<int64_t>(d.tiles_m) * d.tiles_k;
    if (total > INT_MAX) return NF4_ERR_INVALID;
  }
  // Streamed pass: its jobs in the GEMM's order (the sorted descriptors), each
  // problem's ready counters after the work counter and the claim flags; the
  // parts of a fused problem count into the same words.
  StreamJobs sjobs;
  if (streamed) {
    std::memset(&sjobs, 0, sizeof(sjobs));
    sjobs.next = stream_area;
    sjobs.claims = stream_area + 1;
    unsigned int* ready = stream_area + 1 + kStreamClaimWords;
    int items = 0;
    for (size_t i = 0; i < descs.size(); ++i) {
      if (jobs_of[i] < 0) continue;
      // One slab height for all parts of a problem (their counts share the
      // ready words), from the source bytes of a whole row.
      size_t row_bytes = 0;
      for (int q = 0; q < jobs_n[i]; ++q) {
        const F16Job& f = jobs[jobs_of[i] + q];
        row_bytes += static_cast<size_t>(f.N) * (f.mode == kSrcF32 ? 4u : 2u);
      }
      const int slab = slab_rows_for(row_bytes);
      for (int q = 0; q < jobs_n[i]; ++q) {
        const F16Job& f = jobs[jobs_of[i] + q];
        StreamJob& j = sjobs.job[sjobs.n++];
        j.src = f.src;
        j.dst = f.dst;
        j.ready = ready;
        j.mode = f.mode;
        j.M = descs[i].M;
        j.N = f.N;
        j.ldh = f.ldh;
        j.pitch = f.pitch;
        j.item_begin = items;
        j.groups_per_row = f.groups_per_row;
        j.slab_rows = slab;
        items += (j.M + slab - 1) / slab;
      }
      descs[i].ready = ready;
      descs[i].ready_parts = jobs_n[i];
      descs[i].slab_rows = slab;
      ready += (descs[i].M + 255) / 256;
    }
    sjobs.items = items;
  }
  ProblemDesc* ws = static_cast<ProblemDesc*>(workspace);
  for (size_t i = 0; i < descs.size(); i += kDescsPerUpload) {
    const int n = static_cast<int>(std::min<size_t>(kDescsPerUpload, descs.size() - i));
    DescChunk chunk;
    std::memset(&chunk, 0, sizeof(chunk));
    std::memcpy(chunk.d, descs.data() + i, sizeof(ProblemDesc) * n);
    upload_descs_kernel<<<1, 256, 0, st>>>(chunk, ws + i, n);
    if (cudaGetLastError() != cudaSuccess) return NF4_ERR_CUDA;
  }
  if (streamed) {
    // Bookkeeping from zero, then the pass (one block per SM) and the GEMM as
    // its programmatic dependent, which is scheduled as soon as every block of
    // the pass has started and then runs beside it.
    if (cudaMemsetAsync(stream_area, 0, sizeof(unsigned int) * swords, st) != cudaSuccess)
      return NF4_ERR_CUDA;
    int sms = 0;
    int rc = sm_count(&sms);
    if (rc != NF4_OK) return rc;
    // The GEMM's CTAs need nearly all of an SM's shared memory; an SM that runs a
    // block of the pass must already be configured for the largest shared-memory
    // carveout, or the GEMM's CTA could not join the pass's block there.
    static std::once_flag carveout;
    std::call_once(carveout, [] {
      cudaFuncSetAttribute(to_f16_stream_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                           static_cast<int>(cudaSharedmemCarveoutMaxShared));
    });
    to_f16_stream_kernel<<<static_cast<unsigned>(sms), kStreamThreads, 0, st>>>(sjobs);
    if (cudaGetLastError() != cudaSuccess) return NF4_ERR_CUDA;
    SkArgs sk;
    std::memset(&sk, 0, sizeof(sk));
    sk.streamed = 1;
    ProblemDesc unused;
    std::memset(&unused, 0, sizeof(unused));
    if (tiles512)
      return launch_layout<LayoutPreA2>(unused, ws, static_cast<int>(descs.size()),
                                        static_cast<int>(total), &sk, st, /*pdl=*/true);
    return launch_layout<LayoutPreA>(unused, ws, static_cast<int>(descs.size()),
                                     static_cast<int>(total), &sk, st, /*pdl=*/true);
  }
  // The f16 copies, kF16JobsPerLaunch jobs per launch; the GEMM follows the
  // last of them as a programmatic dependent.
  for (size_t i = 0; i < jobs.size(); i += kF16JobsPerLaunch) {
    F16Jobs batch;
    std::memset(&batch, 0, sizeof(batch));
    batch.n = static_cast<int>(std::min<size_t>(kF16JobsPerLaunch, jobs.size() - i));
    int64_t at = 0;
    for (int j = 0; j < batch.n; ++j) {
      batch.job[j] = jobs[i + j];
      const int64_t size = batch.job[j].begin;
      batch.job[j].begin = at;
      at += size;
    }
    batch.end = at;
    const int rc = launch_f16_jobs(batch, st);
    if (rc != NF4_OK) return rc;
  }
  ProblemDesc unused;
  std::memset(&unused, 0, sizeof(unused));
  if (tiles512)
    return launch_layout<LayoutPreA2>(unused, ws, static_cast<int>(descs.size()),
                                      static_cast<int>(total), nullptr, st, /*pdl=*/!jobs.empty());
  return launch_layout<LayoutPreA>(unused, ws, static_cast<int>(descs.size()),
                                   static_cast<int>(total), nullptr, st, /*pdl=*/!jobs.empty());
}

// nf4_problem -> one-part GProblem (its arguments not checked here).
static GProblem from_plain(const nf4_problem& p) {
  GProblem g;
  std::memset(&g, 0, sizeof(g));
  g.part[0].src = p.grad_out;
  g.part[0].dtype = p.go_dtype;
  g.part[0].N = p.N;
  g.nparts = 1;
  g.scales = p.scales;
  g.data = p.data;
  g.out = p.grad_A;
  g.M = p.M;
  g.N = p.N;
  g.K = p.K;
  return g;
}

// nf4_fused_problem -> GProblem, with the rules of nf4_backward_a_fused.
static int from_fused(const nf4_fused_problem& f, GProblem* g) {
  std::memset(g, 0, sizeof(*g));
  if (f.count <= 0 || f.count > kMaxParts || f.parts == nullptr) return NF4_ERR_INVALID;
  if (f.M < 0 || f.K <= 0 || f.K % 64 != 0) return NF4_ERR_INVALID;
  int64_t ntot = 0;
  for (int i = 0; i < f.count; ++i) {
    const nf4_part& q = f.parts[i];
    if (q.go_dtype != NF4_F32 && q.go_dtype != NF4_BF16 && q.go_dtype != NF4_F16)
      return NF4_ERR_INVALID;
    if (q.N <= 0 || q.N % 8 != 0) return NF4_ERR_INVALID;
    g->part[i].src = q.grad_out;
    g->part[i].dtype = q.go_dtype;
    g->part[i].N = q.N;
    ntot += q.N;
  }
  if (ntot > INT_MAX) return NF4_ERR_INVALID;
  g->nparts = f.count;
  g->scales = f.scales;
  g->data = f.data;
  g->out = f.grad_x;
  g->M = f.M;
  g->N = static_cast<int>(ntot);
  g->K = f.K;
  if (f.M == 0) return NF4_OK;
  if (f.scales == nullptr || f.data == nullptr || f.grad_x == nullptr) return NF4_ERR_INVALID;
  for (int i = 0; i < f.count; ++i) {
    if (f.parts[i].grad_out == nullptr) return NF4_ERR_INVALID;
    if (!aligned(f.parts[i].grad_out, 16)) return NF4_ERR_ALIGN;
  }
  if (!aligned(f.grad_x, 16) || !aligned(f.data, 16) || !aligned(f.scales, 4)) return NF4_ERR_ALIGN;
  return NF4_OK;
}
}  // namespace nf4

extern "C" size_t nf4_backward_a_batched_ws_bytes(const nf4_problem* problems, int count) {
  if (count <= 0 || problems == nullptr) return 0;
  std::vector<GProblem> g(count);
  for (int i = 0; i < count; ++i) g[i] = from_plain(problems[i]);
  return grouped_ws_bytes(g.data(), count);
}

extern "C" int nf4_backward_a_batched_ws(const nf4_problem* problems, int count, void* workspace,
                                         size_t workspace_bytes, void* stream) {
  if (count < 0 || (count > 0 && problems == nullptr)) return NF4_ERR_INVALID;
  std::vector<GProblem> g(count);
  for (int i = 0; i < count; ++i) {
    const nf4_problem& p = problems[i];
    const int rc = check_problem(p.grad_out, p.go_dtype, p.scales, p.data, p.grad_A, p.M, p.N, p.K);
    if (rc != NF4_OK) return rc;
    g[i] = from_plain(p);
  }
  return grouped_ws(g.data(), count, workspace, workspace_bytes, as_stream(stream));
}

extern "C" size_t nf4_backward_a_fused_batched_ws_bytes(const nf4_fused_problem* problems,
                                                        int count) {
  if (count <= 0 || problems == nullptr) return 0;
  std::vector<GProblem> g(count);
  for (int i = 0; i < count; ++i)
    if (from_fused(problems[i], &g[i]) != NF4_OK) return 0;
  return grouped_ws_bytes(g.data(), count);
}

extern "C" int nf4_backward_a_fused_batched(const nf4_fused_problem* problems, int count,
                                            void* workspace, size_t workspace_bytes,
                                            void* stream) {
  if (count < 0 || (count > 0 && problems == nullptr)) return NF4_ERR_INVALID;
  std::vector<GProblem> g(count);
  for (int i = 0; i < count; ++i) {
    const int rc = from_fused(problems[i], &g[i]);
    if (rc != NF4_OK) return rc;
  }
  return grouped_ws(g.data(), count, workspace, workspace_bytes, as_stream(stream));
}

#ifdef NF4_PROGRESS
extern "C" int nf4_debug_set_progress(void* buf) {
  unsigned int* p = static_cast<unsigned int*>(buf);
  return cudaMemcpyToSymbol(g_progress, &p, sizeof(p)) == cudaSuccess ? NF4_OK : NF4_ERR_CUDA;
}
#endif

#ifdef NF4_TRACE
extern "C" int nf4_debug_timeouts(unsigned int* out, int max_entries) {
  unsigned int n = 0;
  if (cudaMemcpyFromSymbol(&n, g_timeout_count, sizeof(n)) != cudaSuccess) return -1;
  const int k = static_cast<int>(n < 256u ? n : 256u) < max_entries ? static_cast<int>(n < 256u ? n : 256u)
                                                                    : max_entries;
  if (k > 0 && cudaMemcpyFromSymbol(out, g_timeout_log, sizeof(unsigned int) * 4 * k) != cudaSuccess)
    return -1;
  return static_cast<int>(n);
}

extern "C" int nf4_debug_set_trace(void* buf) {
  unsigned long long* p = static_cast<unsigned long long*>(buf);
  return cudaMemcpyToSymbol(g_trace, &p, sizeof(p)) == cudaSuccess ? NF4_OK : NF4_ERR_CUDA;
}
#endif

// ------------------------------------------------------------------ watchdog self-test
// One CTA whose waits cannot be satisfied: thread 0 waits on an mbarrier that
// nothing arrives on, with a short limit, so it gives up, records the timeout
// (status word and site) and raises the CTA's abort flag; thread 32 waits on a
// second such barrier with the normal limit and must return as soon as it sees
// the flag (without recording a second site).  Both then exit: the context
// stays usable.  `where` receives the first barrier's shared-memory address
// and whether the second wait returned without a completed phase.
__global__ void wait_selftest_kernel(long long limit, unsigned int* where) {
  __shared__ __align__(8) unsigned long long bars[2];
  __shared__ int abort_word;
  volatile int* abort_flag = &abort_word;
  const uint32_t b0 = smem_addr(&bars[0]), b1 = smem_addr(&bars[1]);
  if (threadIdx.x == 0) {
    mbar_init(b0, 1);
    mbar_init(b1, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const bool ok = mbar_wait(b0, 0, abort_flag, limit);
    where[0] = b0;
    where[1] = ok ? 1u : 0u;
  } else if (threadIdx.x == 32) {
    where[2] = mbar_wait(b1, 0, abort_flag) ? 1u : 0u;
  }
  __syncthreads();
}

extern "C" int nf4_watchdog_selftest(long long limit_cycles, unsigned int* where, void* stream) {
  if (limit_cycles < 1000 || limit_cycles > kWaitLimitCycles || where == nullptr ||
      !aligned(where, 4))
    return NF4_ERR_INVALID;
  wait_selftest_kernel<<<1, 64, 0, as_stream(stream)>>>(limit_cycles, where);
  return launch_status();
}

extern "C" int nf4_check_error(void* stream) {
  return nf4_check_error_site(stream, nullptr);
}

extern "C" int nf4_check_error_site(void* stream, unsigned int* site) {
  if (site != nullptr) std::memset(site, 0, 4 * sizeof(unsigned int));
  if (cudaStreamSynchronize(as_stream(stream)) != cudaSuccess) return NF4_ERR_CUDA;
  unsigned int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_status, sizeof(v)) != cudaSuccess) return NF4_ERR_CUDA;
  if (v != 0) {
    unsigned int where[4] = {0, 0, 0, 0};
    cudaMemcpyFromSymbol(where, g_timeout_site, sizeof(where));
    if (site != nullptr) std::memcpy(site, where, sizeof(where));
    const unsigned int zero[4] = {0, 0, 0, 0};
    cudaMemcpyToSymbol(g_status, zero, sizeof(unsigned int));
    cudaMemcpyToSymbol(g_timeout_site, zero, sizeof(zero));
    return NF4_ERR_TIMEOUT;
  }
  return cudaGetLastError() == cudaSuccess ? NF4_OK : NF4_ERR_CUDA;
}

// ------------------------------------------------------------------ grouped launch without allocation
// Some callers cannot allocate device memory for the grouped launch's
// workspace: code that runs under a caching allocator it must not re-enter, in a
// stream-ordered region where cudaMalloc would synchronise the device, or in a
// process whose memory is fully reserved up front.  For them the descriptors
// live in this file-scope device array instead.  It is reserved on every GPU
// that loads the library, for the life of the process, and shared by every
// call of nf4_backward_a_batched_noalloc on that GPU.
namespace nf4 {
constexpr int kNoAllocMaxProblems = 256;
constexpr size_t kNoAllocBytes = kNoAllocMaxProblems * sizeof(ProblemDesc);  // 160 KiB
static __device__ __align__(256) unsigned char g_noalloc_descs[kNoAllocBytes];

// Device address of g_noalloc_descs on the current device, looked up once per
// device.  In host code the array's name is only a host-side stand-in for the
// symbol; cudaGetSymbolAddress gives the address a kernel may use.
static int noalloc_descs(ProblemDesc** out) {
  static ProblemDesc* addr[64] = {};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return NF4_ERR_CUDA;
  std::lock_guard<std::mutex> lock(mu);
  if (addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_descs) != cudaSuccess || p == nullptr)
      return NF4_ERR_CUDA;
    addr[dev] = static_cast<ProblemDesc*>(p);
  }
  *out = addr[dev];
  return NF4_OK;
}
}  // namespace nf4

extern "C" int nf4_backward_a_batched_noalloc(const nf4_problem* problems, int count,
                                              void* stream) {
  if (count < 0 || (count > 0 && problems == nullptr)) return NF4_ERR_INVALID;
  if (count > kNoAllocMaxProblems) return NF4_ERR_WORKSPACE;
  for (int i = 0; i < count; ++i) {
    const nf4_problem& p = problems[i];
    if (p.go_dtype == NF4_F16) return NF4_ERR_INVALID;  // single calls only
    const int rc = check_problem(p.grad_out, p.go_dtype, p.scales, p.data, p.grad_A, p.M, p.N, p.K);
    if (rc != NF4_OK) return rc;
  }
  cudaStream_t st = as_stream(stream);
  // Problems that need the GEMM, longest tiles first (stable), as the grouped
  // entry point orders them; no heap memory is used on the host either.
  int order[kNoAllocMaxProblems];
  int stages[kNoAllocMaxProblems];
  int n = 0;
  const int small_max = small_m::g_max_m.load();
  for (int i = 0; i < count; ++i) {
    const nf4_problem& p = problems[i];
    if (p.M == 0) continue;
    if (p.N == 0) {
      if (cudaMemsetAsync(p.grad_A, 0, sizeof(float) * static_cast<size_t>(p.M) * p.K, st) !=
          cudaSuccess)
        return NF4_ERR_CUDA;
      continue;
    }
    if (p.M <= small_max) {
      const int rc = small_m::run(p.grad_out, p.go_dtype, p.scales, p.data, p.grad_A, p.M, p.N,
                                  p.K, st);
      if (rc != NF4_OK) return rc;
      continue;
    }
    const int ns = (p.N + BN - 1) / BN;
    int j = n++;
    while (j > 0 && stages[j - 1] < ns) {
      order[j] = order[j - 1];
      stages[j] = stages[j - 1];
      --j;
    }
    order[j] = i;
    stages[j] = ns;
  }
  if (n == 0) return NF4_OK;
  ProblemDesc* ws = nullptr;
  int rc = noalloc_descs(&ws);
  if (rc != NF4_OK) return rc;
  // Every descriptor the GEMM reads is written here, in stream order before it,
  // so nothing left in the array by an earlier call is ever used.
  DescChunk chunk;
  int64_t total = 0;
  for (int i = 0; i < n; i += kDescsPerUpload) {
    const int m = std::min(kDescsPerUpload, n - i);
    std::memset(&chunk, 0, sizeof(chunk));
    for (int j = 0; j < m; ++j) {
      const nf4_problem& p = problems[order[i + j]];
      ProblemDesc& d = chunk.d[j];
      rc = fill_desc(&d, p.grad_out, p.go_dtype, p.scales, p.data, p.grad_A, p.M, p.N, p.K);
      if (rc != NF4_OK) return rc;
      d.tile_begin = static_cast<int>(total);
      total += static_cast<int64_t>(d.tiles_m) * d.tiles_k;
      if (total > INT_MAX) return NF4_ERR_INVALID;
    }
    upload_descs_kernel<<<1, 256, 0, st>>>(chunk, ws + i, m);
    if (cudaGetLastError() != cudaSuccess) return NF4_ERR_CUDA;
  }
  ProblemDesc unused;
  std::memset(&unused, 0, sizeof(unused));
  bool all_bf16 = true;
  for (int i = 0; i < n; ++i) all_bf16 = all_bf16 && problems[order[i]].go_dtype == NF4_BF16;
  return launch(unused, ws, n, static_cast<int>(total), all_bf16, st);
}

// ------------------------------------------------------------------ dense GemmBackwardB
namespace nf4 {
namespace dense {

// Pairs of CTAs of the kernel that fit on the current device at once (also
// sets its shared-memory limit).
static int max_pairs(int* out) {
  static int cached[64] = {};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return NF4_ERR_CUDA;
  std::lock_guard<std::mutex> lock(mu);
  if (cached[dev] == 0) {
    if (cudaFuncSetAttribute(backward_b_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kSmemBytes) != cudaSuccess)
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
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int clusters = 0;
    if (cudaOccupancyMaxActiveClusters(&clusters, backward_b_kernel, &cfg) != cudaSuccess ||
        clusters <= 0)
      clusters = sms / 2;
    cached[dev] = clusters;
  }
  *out = cached[dev];
  return NF4_OK;
}

// Splits of the token range: one when the tiles fill the pairs, else as many as
// keep every pair busy, each split at least 8 stages (512 tokens) long.
static int plan_splits(int tiles, int stages, int pairs) {
  if (tiles <= 0 || stages <= 0 || pairs <= tiles) return 1;
  const int s = std::min(pairs / tiles, stages / 8);
  return s > 1 ? s : 1;
}

static inline int tiles_of(int extent, int tile) { return (extent + tile - 1) / tile; }

}  // namespace dense
}  // namespace nf4

extern "C" int nf4_gemm_backward_b_splits(int M, int K, int N, int pairs) {
  if (M < 0 || K <= 0 || N <= 0 || pairs <= 0) return -1;
  if (M == 0) return 1;
  return dense::plan_splits(dense::tiles_of(K, dense::kTileK) * dense::tiles_of(N, dense::kTileN),
                            dense::tiles_of(M, dense::kTok), pairs);
}

extern "C" size_t nf4_gemm_backward_b_ws_bytes(int M, int K, int N) {
  if (M <= 0 || K <= 0 || N <= 0) return 0;
  int pairs = 0;
  if (dense::max_pairs(&pairs) != NF4_OK) return 0;
  const int splits = nf4_gemm_backward_b_splits(M, K, N, pairs);
  if (splits <= 1) return 0;
  return sizeof(float) * static_cast<size_t>(splits) *
         static_cast<size_t>(dense::tiles_of(K, dense::kTileK) * dense::kTileK) *
         static_cast<size_t>(N);
}

extern "C" int nf4_gemm_backward_b(const void* A, const void* grad_C, int dtype, float* grad_B,
                                   int M, int K, int N, void* workspace, size_t workspace_bytes,
                                   void* stream) {
  using namespace nf4::dense;
  if (dtype != NF4_BF16 && dtype != NF4_F16) return NF4_ERR_INVALID;
  if (M < 0 || K <= 0 || N <= 0 || K % 8 != 0 || N % 8 != 0) return NF4_ERR_INVALID;
  if (grad_B == nullptr) return NF4_ERR_INVALID;
  if (!aligned(grad_B, 16)) return NF4_ERR_ALIGN;
  cudaStream_t st = as_stream(stream);
  if (M == 0) {
    return cudaMemsetAsync(grad_B, 0, sizeof(float) * static_cast<size_t>(K) * N, st) == cudaSuccess
               ? NF4_OK
               : NF4_ERR_CUDA;
  }
  if (A == nullptr || grad_C == nullptr) return NF4_ERR_INVALID;
  if (!aligned(A, 16) || !aligned(grad_C, 16)) return NF4_ERR_ALIGN;
  int pairs = 0;
  int rc = max_pairs(&pairs);
  if (rc != NF4_OK) return rc;
  Args a;
  std::memset(&a, 0, sizeof(a));
  a.tiles_k = tiles_of(K, kTileK);
  a.tiles_n = tiles_of(N, kTileN);
  a.stages = tiles_of(M, kTok);
  a.splits = nf4_gemm_backward_b_splits(M, K, N, pairs);
  const int kp = a.tiles_k * kTileK;
  const size_t slice = sizeof(float) * static_cast<size_t>(kp) * static_cast<size_t>(N);
  // The split needs its partial sums; with less workspace, fewer splits.
  if (a.splits > 1 && (workspace == nullptr || !aligned(workspace, 256)))
    a.splits = 1;
  while (a.splits > 1 && workspace_bytes < slice * static_cast<size_t>(a.splits)) --a.splits;
  const int64_t items = static_cast<int64_t>(a.tiles_k) * a.tiles_n * a.splits;
  if (items > INT_MAX) return NF4_ERR_INVALID;
  a.items = static_cast<int>(items);
  a.kp = a.splits > 1 ? kp : 0;
  a.idesc = idesc_f16_f32(2 * kRowsCta, kTileN, /*A MN-major*/ 1, /*B MN-major*/ 1,
                          dtype == NF4_BF16 ? 1u : 0u);
  const CUtensorMapDataType t16 =
      dtype == NF4_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  float* out = a.splits > 1 ? static_cast<float*>(workspace) : grad_B;
  const uint64_t out_rows = a.splits > 1 ? static_cast<uint64_t>(a.splits) * kp
                                         : static_cast<uint64_t>(K);
  if (!encode_2d(&a.tm_a, t16, A, static_cast<uint64_t>(K), static_cast<uint64_t>(M),
                 static_cast<uint64_t>(K) * 2, 64, kTok, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_2d(&a.tm_c, t16, grad_C, static_cast<uint64_t>(N), static_cast<uint64_t>(M),
                 static_cast<uint64_t>(N) * 2, 64, kTok, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_2d(&a.tm_out, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, out, static_cast<uint64_t>(N),
                 out_rows, static_cast<uint64_t>(N) * 4, kEpiCols, 32,
                 CU_TENSOR_MAP_SWIZZLE_64B))
    return NF4_ERR_CUDA;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(static_cast<unsigned>(2 * std::min(a.items, pairs)), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, backward_b_kernel, a) != cudaSuccess) return NF4_ERR_CUDA;
  if (a.splits > 1) {
    int sms = 0;
    rc = sm_count(&sms);
    if (rc != NF4_OK) return rc;
    const int64_t work = static_cast<int64_t>(K) * (N / 4);
    const int64_t blocks = std::min<int64_t>((work + 255) / 256, static_cast<int64_t>(sms) * 8);
    reduce_splits_kernel<<<static_cast<unsigned>(blocks), 256, 0, st>>>(
        static_cast<const float*>(workspace), grad_B, a.splits, K, N, kp);
  }
  return launch_status();
}
