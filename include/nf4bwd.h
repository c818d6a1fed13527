/*
 * nf4bwd.h -- C ABI of libnf4bwd.so, the NF4-dequant-fused backward-A GEMM
 * for GB300 (sm_103a).
 *
 * The operation (page "aprender-gpu 0.32.0 -- src/kernels/backward/
 * nf4_tensor_core.rs", struct doc comment of Nf4TensorCoreGemmBackwardAKernel):
 *
 *     grad_A[M x K] = grad_out[M x N] @ dequant(B_nf4[K x N])^T
 *
 * N is the shared (contraction) dimension, K the output dimension; B_nf4 is the
 * frozen 4-bit NormalFloat weight of a linear layer with K inputs and N outputs.
 *
 * Conventions for every entry point below
 *   - All array pointers are DEVICE pointers owned by the caller.  The library
 *     allocates nothing, keeps no reference after the call returns and never
 *     frees caller memory.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *     Work is enqueued asynchronously on it; the call returns before the GPU
 *     finishes.  Inputs must stay valid until the stream reaches the work.
 *   - The return value is an nf4_status.  Argument errors are detected on the
 *     host before anything is enqueued, and then nothing is written.
 *   - Kernel faults are not detected by the call itself; a bounded wait inside
 *     a kernel that gives up (no progress for 1 s) sets a device status word
 *     that nf4_check_error() reports as NF4_ERR_TIMEOUT.
 *
 * Data layout (page above, build_ptx "PHASE 2: Dequant B_nf4"):
 *   scales   fp32 [N][K/64]   absmax of the 64-element K-block b of column n
 *   data     u8   [N][K/2]    codes of column n, K contiguous: element (k, n)
 *                             is nibble (k % 2) of byte n*(K/2) + k/2, low
 *                             nibble = even k
 *   grad_out [M][N] row-major, fp32 or bf16
 *   grad_A   fp32 [M][K] row-major, overwritten (not accumulated into)
 *
 * Arithmetic (same page, build_ptx phases 1-3): every dequantised weight is
 * f16_rn(f32(scale * codebook[code])); grad_out is rounded to f16 (bf16 input:
 * widened exactly to f32 first); products of the f16 operands are summed in
 * fp32 by the tensor cores (tcgen05, accumulator in tensor memory).
 */
#ifndef NF4BWD_H
#define NF4BWD_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum nf4_status {
  NF4_OK = 0,
  NF4_ERR_INVALID = 1, /* null pointer, negative size, K % 64 != 0, N not a multiple of
                          the row alignment (4 for fp32 grad_out, 8 for bf16), ... */
  NF4_ERR_ALIGN = 2,   /* a pointer is not 16-byte aligned (scales: 4-byte) */
  NF4_ERR_CUDA = 3,    /* a CUDA runtime call or a kernel launch failed */
  NF4_ERR_TIMEOUT = 4, /* a kernel's bounded wait gave up (reported by nf4_check_error) */
  NF4_ERR_WORKSPACE = 5 /* workspace missing, misaligned or too small */
} nf4_status;

/* Type of grad_out.  NF4_F16 is already the GEMM's operand type (no rounding
 * step); it is accepted by nf4_backward_a_ex and nf4_backward_a_ws only. */
typedef enum nf4_dtype { NF4_F32 = 0, NF4_BF16 = 1, NF4_F16 = 2 } nf4_dtype;

/* Version of this ABI (incremented on any incompatible change). */
int nf4_abi_version(void);

/* Human-readable name of a status code (static string, never NULL). */
const char* nf4_status_string(int status);

/*
 * Quantise a dense fp32 weight B [K][N] (row-major) to NF4: for every column n
 * and 64-element K-block b, scales[n][b] = max |B[k][n]| over the block, and
 * each element gets the code of the nearest codebook entry to B/scale (f32
 * differences, ties to the lower code; an all-zero block gets scale 0 and code
 * 7).  The pages fix the packed layout (page above, build_ptx "PHASE 2") but
 * not the quantiser; this is blockwise absmax NormalFloat4 quantisation as in
 * Dettmers et al., "QLoRA" (2023).
 *   B       [K*N] fp32, 16-byte aligned not required (4-byte)
 *   data    [N*K/2] bytes, 16-byte aligned; scales [N*K/64] fp32, 4-byte aligned
 *   K       positive multiple of 64; N positive
 */
int nf4_quantize(const float* B, int K, int N, uint8_t* data, float* scales, void* stream);

/*
 * Dequantise to f16, transposed: bt[n*K + k] = f16 bits of
 * f16_rn(f32(scales[n][k/64] * codebook[code(k, n)])) (page above, build_ptx
 * "PHASE 2").  Runs the same device routine that the GEMM's producer warps use
 * to build the B^T operand, so it exposes their values for bit-exact checks.
 *   bt      [N*K] uint16 (f16 bits), 16-byte aligned
 */
int nf4_dequantize_f16(const float* scales, const uint8_t* data, int K, int N, uint16_t* bt,
                       void* stream);

/*
 * grad_A = grad_out @ dequant(B_nf4)^T with fp32 grad_out (page above, the
 * kernel's parameter list: grad_out_ptr, scales_ptr, data_ptr, grad_a_ptr, m, n,
 * k).  M == 0 enqueues nothing; N == 0 writes zeros into grad_A.
 *   grad_out [M*N] fp32, 16-byte aligned, N % 4 == 0
 *   data     16-byte aligned; scales 4-byte aligned; grad_A [M*K] fp32, 16-byte aligned
 *   K        positive multiple of 64
 */
int nf4_backward_a(const float* grad_out, const float* scales, const uint8_t* data,
                   float* grad_A, int M, int N, int K, void* stream);

/* As nf4_backward_a, with grad_out of type go_dtype (NF4_F32, NF4_BF16 or
 * NF4_F16; bf16 and f16 need N % 8 == 0).  f16 grad_out feeds the pair kernel's
 * TMA-loaded A operand as it is, whatever M (the few-token kernel takes fp32
 * and bf16 only); its result equals nf4_backward_a_ws's without a split for
 * the same values given in fp32 or bf16 (the rounding to f16 then happens first). */
int nf4_backward_a_ex(const void* grad_out, int go_dtype, const float* scales,
                      const uint8_t* data, float* grad_A, int M, int N, int K, void* stream);

/*
 * Bytes of device workspace nf4_backward_a_ws needs for an M x N grad_out on
 * the current device: an f16 copy with rows padded to a multiple of 8 elements
 * (2 * M * ((N + 7) & ~7) bytes, rounded up to 256), then room for the split
 * of a last partial wave of tiles (nf4_split_plan): one flag word and one
 * 256 KiB fp32 partial-sum tile per pair of CTAs the device runs at once.
 * 0 when M or N is not positive.
 */
size_t nf4_backward_a_ws_bytes(int M, int N);

/*
 * As nf4_backward_a_ex, in two launches on `stream`: a streaming pass rounds
 * grad_out to f16 (the rounding the GEMM applies to its A operand anyway: page
 * above, build_ptx "PHASE 1", cvt.rn.f16) into `workspace`, then the GEMM loads
 * its A operand from that copy with TMA instead of converting it in shared
 * memory.  Without a split (nf4_split_plan) the result equals
 * nf4_backward_a_ex's bit for bit; a split tile adds the pairs' fp32 partial
 * sums in pair order, a different but fixed rounding.  The pages have
 * no counterpart of the split: it trades 6 (fp32) or 4 (bf16) bytes of HBM
 * traffic per grad_out element for shared-memory bandwidth inside the GEMM.
 *   workspace        caller-owned device memory, 256-byte aligned, at least
 *                    nf4_backward_a_ws_bytes(M, N) bytes; overwritten; must not
 *                    be used by anything else until the stream has run the call
 *   workspace_bytes  its size; smaller than the f16 copy, NULL or misaligned
 *                    returns NF4_ERR_WORKSPACE and enqueues nothing; room for
 *                    the f16 copy only runs every tile whole (no split)
 * M at most the few-token limit (nf4_set_small_m_max), M == 0 and N == 0 take
 * the same paths as nf4_backward_a_ex and do not touch the workspace (it may
 * then be NULL).  With NF4_F16 grad_out there is no pre-pass: the GEMM reads
 * grad_out directly and the workspace's copy region goes unused.
 */
int nf4_backward_a_ws(const void* grad_out, int go_dtype, const float* scales,
                      const uint8_t* data, float* grad_A, int M, int N, int K, void* workspace,
                      size_t workspace_bytes, void* stream);

/*
 * The forward product C[M x N] = A[M x K] @ dequant(B_nf4[K x N]), contracted
 * over K (page above, module header: the backward kernel is described there as
 * the transposed counterpart of a forward NF4 tensor-core GEMM over the same
 * NF4 layout: data [N][K/2], scales [N][K/64]).  Same arithmetic as
 * the backward: A rounded to f16 (RNE), dequant(B)[k,n] =
 * f16(f32(scale[n][k/64] * codebook[code])), f32 accumulation, C overwritten.
 * Two launches on `stream`, as nf4_backward_a_ws: an f16 pre-pass of A into
 * `workspace` (none for NF4_F16 A), then the pair kernel with the dequantised
 * weight as its K-major B operand (256 columns n per pair tile, 64 k per
 * stage).  No counterpart kernel on the pages.
 *   A       [M*K] of type a_dtype (NF4_F32, NF4_BF16 or NF4_F16), 16-byte aligned
 *   data    [N][K/2] bytes, 16-byte aligned; scales [N][K/64] fp32, 4-byte aligned
 *   C       [M*N] fp32, 16-byte aligned, N % 4 == 0 (its rows are TMA-stored)
 *   K       positive multiple of 64; M == 0 or N == 0 enqueue nothing
 *   workspace, workspace_bytes: as nf4_backward_a_ws, at least
 *           nf4_forward_ws_bytes(M, K) bytes for the split of a last partial
 *           wave, at least the f16 copy (2 * M * K bytes) in any case
 * Returns NF4_ERR_INVALID, NF4_ERR_ALIGN or NF4_ERR_WORKSPACE (nothing
 * enqueued) for arguments outside these rules.
 */
size_t nf4_forward_ws_bytes(int M, int K);
int nf4_forward_ws(const void* A, int a_dtype, const float* scales, const uint8_t* data, float* C,
                   int M, int N, int K, void* workspace, size_t workspace_bytes, void* stream);

/* One projection of a fused call (nf4_backward_a_fused). */
typedef struct nf4_part {
  const void* grad_out; /* [M][N] of type go_dtype, 16-byte aligned */
  int go_dtype;         /* NF4_F32, NF4_BF16 or NF4_F16 */
  int N;                /* the projection's output width, a positive multiple of 8 */
} nf4_part;

/*
 * Input gradient of a layer input shared by several projections, summed in
 * one GEMM:
 *
 *     grad_x[M x K] = sum_p grad_out_p[M x N_p] @ dequant(B_p[K x N_p])^T
 *
 * The page's doc comment counts 7 backward projections per layer (page above,
 * struct doc comment); q, k and v read the same layer input, as do gate and up
 * (the same page's Qwen-dimension test: q/k/v and gate/up share the input width
 * K), so their input gradients add.  Summing them over the concatenated shared
 * dimension N = sum N_p in one accumulator replaces count separate grad_A
 * results and their addition.  The pages do not spell the fusion out; this is
 * the sum of the backward-A products, each with the arithmetic of
 * nf4_backward_a_ws (operands rounded to f16, f32 accumulation).  Two launches
 * on `stream`: a pass writes each part's grad_out, rounded to f16, into its
 * columns of one A operand in `workspace`, then the pair kernel runs the
 * single problem M x N x K (every M: no few-token path).  The result equals,
 * bit for bit, nf4_backward_a_ws on the column-wise concatenation of the
 * grad_out parts with the stacked weight.
 *   parts    HOST array of `count` parts (1..64), read before the call returns
 *   scales, data  the parts' NF4 weights stacked along N in part order:
 *            data [sum N_p][K/2], scales [sum N_p][K/64] (rows of each
 *            weight's data and scales concatenated; this is what nf4_quantize
 *            gives for the dense weights concatenated along N, since every
 *            64-element block lies within one column)
 *   grad_x   [M][K] fp32, 16-byte aligned, overwritten
 *   K        positive multiple of 64; M == 0 enqueues nothing
 *   workspace, workspace_bytes  as nf4_backward_a_ws with N = sum N_p: at least
 *            the f16 copy (2 * M * sum N_p bytes); nf4_backward_a_ws_bytes(M,
 *            sum N_p) bytes allow the split of a last partial wave
 * Returns NF4_ERR_INVALID, NF4_ERR_ALIGN or NF4_ERR_WORKSPACE (nothing
 * enqueued) for arguments outside these rules.
 */
int nf4_backward_a_fused(const nf4_part* parts, int count, const float* scales,
                         const uint8_t* data, float* grad_x, int M, int K, void* workspace,
                         size_t workspace_bytes, void* stream);

/* One problem of nf4_backward_a_fused_batched: the arguments of one
 * nf4_backward_a_fused call. */
typedef struct nf4_fused_problem {
  const nf4_part* parts; /* HOST array of `count` parts (1..8), read before the call returns */
  int count;
  const float* scales;   /* the parts' weights stacked along N: [sum N_p][K/64] */
  const uint8_t* data;   /* [sum N_p][K/2] */
  float* grad_x;         /* [M][K], overwritten */
  int M, K;
} nf4_fused_problem;

/* Bytes of workspace nf4_backward_a_fused_batched needs for these problems
 * (descriptors, one f16 copy [M][sum N_p] per problem, and the bookkeeping of
 * the pass beside the GEMM); 0 for count <= 0 or a problem outside the rules. */
size_t nf4_backward_a_fused_batched_ws_bytes(const nf4_fused_problem* problems, int count);

/*
 * Many fused problems in one grouped launch: the pre-converted grouped path of
 * nf4_backward_a_batched_ws over problems that are each a sibling-projection
 * sum (nf4_backward_a_fused), e.g. the q/k/v and gate/up input gradients of
 * every layer of a model plus its unfused o and down projections (one part
 * each) in one call.  Every part's grad_out is rounded to f16 into its columns
 * of its problem's copy in the workspace, by the pass that runs beside the GEMM
 * (or before it, when the workspace has room for the descriptors and copies
 * only); each problem's grad_x equals, bit for bit, what nf4_backward_a_fused
 * gives for it without a split.  Every problem runs on the pair kernel,
 * whatever its M.  No counterpart on the pages.
 *   workspace  caller-owned device memory, 256-byte aligned,
 *              nf4_backward_a_fused_batched_ws_bytes(problems, count) bytes;
 *              smaller than the descriptors and copies, NULL or misaligned
 *              returns NF4_ERR_WORKSPACE and enqueues nothing
 * Returns NF4_ERR_INVALID or NF4_ERR_ALIGN (nothing enqueued) for a problem
 * outside the rules of nf4_backward_a_fused or with more than 8 parts.
 */
int nf4_backward_a_fused_batched(const nf4_fused_problem* problems, int count, void* workspace,
                                 size_t workspace_bytes, void* stream);

/*
 * Tokens per pair tile, 256 or 512, that the pre-converted kernel uses for an
 * M x N x K problem run by `pairs` pairs of CTAs (pure host computation).  A
 * 512-token tile issues two M = 256 MMA blocks against each dequantised B^T
 * stage, halving the dequantisation per MMA, but its two accumulators fill
 * tensor memory, so its epilogue does not overlap the next tile and its tiles
 * are never split.  512 when the problem has at least 8 stages (N >= 449) and
 * at least pairs / 2 such tiles; 256 otherwise (a rule from measurements;
 * can_split is accepted for the split-aware choice and currently unused).
 * -1 for a non-positive argument.
 */
int nf4_tile_rows(int M, int N, int K, int pairs, int can_split);

/*
 * Force the pre-converted kernel's tile (256 or 512 tokens) for calls made
 * after this returns, or 0 to choose by nf4_tile_rows (the default).  Returns
 * the previous setting, or -1 (nothing changed) for another value.
 * Process-wide.  Both tiles give the same results bit for bit.
 */
int nf4_set_tile_rows(int rows);

/*
 * The split plan of nf4_backward_a_ws, as pure host computations (no device is
 * touched), for `tiles` pair tiles (256 tokens x 256 output columns) of
 * `stages` 64-wide stages of N each, run by `pairs` pairs of CTAs.  Whole waves
 * of tiles stay whole (tiles [0, dp_tiles), round-robin); when splitting the
 * last, partial wave saves every pair at least 40 stages (stages * (pairs -
 * rem) >= 40 * pairs, rem = tiles % pairs), its sk_tiles = rem tiles are split
 * by stages, one contiguous run of their stages per pair.  Returns -1 for a
 * non-positive count or a NULL output.
 */
int nf4_split_plan(int tiles, int stages, int pairs, int* dp_tiles, int* sk_tiles);

/*
 * Item k (k = 0, 1, ...) of pair `pair` under that plan, in the order the pair
 * runs them: item[0] the tile, [item[1], item[2]) its stages, and for the
 * first stages of a split tile the range item[3] .. item[4] of pairs whose
 * partial sums the pair adds before storing the tile: every pair of the range
 * that holds stages of split tiles (item[4] < item[3]: none).  Returns 1, 0 when the pair has
 * no item k, -1 for invalid arguments.
 */
int nf4_split_item(int tiles, int stages, int pairs, int pair, int k, int* item);

/*
 * Few-token path.  A call of nf4_backward_a / nf4_backward_a_ex with M at most
 * this limit runs a kernel built for small M: the weight is streamed once
 * (256 output columns per CTA, all tokens at once) and the shared dimension N
 * is split over a cluster of up to 16 CTAs whose partial sums are added in a
 * fixed order (the result is deterministic, but its rounding differs from the
 * general kernel's).  The default limit is 64, the
 * largest allowed; 0 sends every M to the general kernel.  Returns the previous
 * limit.  Process-wide; takes effect for calls made after it returns.
 */
int nf4_set_small_m_max(int m_max);

/*
 * The small-M path's choice of cluster size S for an N x K weight, as a pure
 * host computation (no device is touched): `sms` SMs holding `cta_slots` CTAs
 * at once in all, so that cta_slots / S clusters of size S fit.  Writes to
 * *per_out the number of 64-wide N stages of each cluster rank and returns S
 * (1..16), or -1 for a non-positive argument or a NULL per_out.  The launch
 * makes the same choice from the device's real cluster occupancy.
 */
int nf4_small_m_split(int N, int K, int sms, int cta_slots, int* per_out);

/* One projection of a grouped launch. */
typedef struct nf4_problem {
  const void* grad_out; /* [M][N], type go_dtype */
  int go_dtype;         /* NF4_F32 or NF4_BF16; NF4_F16 in nf4_backward_a_batched_ws only */
  const float* scales;  /* [N][K/64] */
  const uint8_t* data;  /* [N][K/2] */
  float* grad_A;        /* [M][K], overwritten */
  int M, N, K;
} nf4_problem;

/* Bytes of device workspace nf4_backward_a_batched needs for `count` problems. */
size_t nf4_backward_a_batched_workspace(int count);

/*
 * Grouped backward-A over `count` independent projections in one persistent
 * launch (the page's doc comment counts 28 layers x 7 projections = 196
 * backward projections per training step).  Every problem follows the rules of
 * nf4_backward_a_ex.  `problems` is a HOST array, read before the call returns.
 * `workspace` is caller-owned device memory of at least
 * nf4_backward_a_batched_workspace(count) bytes, 256-byte aligned.  The call
 * enqueues, on `stream`, small kernels that write the per-problem descriptors
 * (tensor maps, pointers, sizes) into it -- the descriptors travel as kernel
 * parameters, so nothing on the host has to outlive the call -- and then the
 * GEMM kernel that reads them.  The workspace must not be reused by another
 * call until this one has run.  Problems with M at most the few-token limit
 * (nf4_set_small_m_max) are not part of the grouped launch: each runs as its
 * own launch of the few-token kernel, so every problem's grad_A equals, bit
 * for bit, what a single call gives.
 */
int nf4_backward_a_batched(const nf4_problem* problems, int count, void* workspace,
                           size_t workspace_bytes, void* stream);

/*
 * Bytes of workspace nf4_backward_a_batched_ws needs for these problems: the
 * descriptors (the same as nf4_backward_a_batched's, rounded up to 256), an
 * f16 copy of every fp32 or bf16 grad_out (2 * M * ((N + 7) & ~7) bytes each,
 * rounded up to 256), and, when at most 256 problems have such a copy, the
 * bookkeeping of the pass that writes the copies beside the GEMM (4 bytes per
 * 256-row block of each such problem plus 1028, rounded up to 256).  `problems`
 * is a host array; 0 for count <= 0.
 */
size_t nf4_backward_a_batched_ws_bytes(const nf4_problem* problems, int count);

/*
 * The grouped launch of the pre-converted path (see nf4_backward_a_ws): every
 * fp32 or bf16 grad_out is rounded to f16 into the workspace, and one
 * persistent launch of the pair kernel with TMA-loaded A operands runs all
 * problems' tiles (longest first).  With the full workspace the rounding pass
 * runs BESIDE the GEMM: one block of it per SM converts slabs of rows (8 to 64
 * rows, fewer for wide rows) in the GEMM's order and counts each finished slab
 * into its 256-row block's ready
 * word; the GEMM (a programmatic dependent of the pass, so it starts as soon
 * as the pass has) waits for a block's count before its first copy from it.
 * With room for the descriptors and copies only, the passes run first and the
 * GEMM follows the last of them.  The results are the same.  NF4_F16 grad_out is accepted and
 * read in place.  Few-token problems (M at most nf4_set_small_m_max, fp32 or
 * bf16) run as their own launches of the few-token kernel, as in
 * nf4_backward_a_batched.  Each problem's grad_A equals, bit for bit, what
 * nf4_backward_a_ws gives for it without a split (tiles are never split
 * here).  No counterpart on the pages.
 *   workspace  caller-owned device memory, 256-byte aligned,
 *              nf4_backward_a_batched_ws_bytes(problems, count) bytes; smaller
 *              than the descriptors and copies, NULL or misaligned returns
 *              NF4_ERR_WORKSPACE and enqueues nothing; must not be reused until
 *              the stream has run the call
 */
int nf4_backward_a_batched_ws(const nf4_problem* problems, int count, void* workspace,
                              size_t workspace_bytes, void* stream);

/*
 * Grouped backward-A that allocates nothing.  The pages have no counterpart of
 * this entry point: it exists for callers that cannot allocate device memory
 * for the workspace of nf4_backward_a_batched -- code running inside a caching
 * allocator it must not re-enter, inside a stream-ordered region where
 * cudaMalloc would synchronise the device, or in a process whose device memory
 * is all reserved up front.
 *
 * Same problems, rules and results as nf4_backward_a_batched (few-token
 * problems included), but the
 * per-problem descriptors go to a fixed array inside the library (a
 * file-scope device array of 160 KiB, reserved on every GPU that loads the
 * library until the process exits), so the call takes no workspace.
 *   count      at most 256 problems; more returns NF4_ERR_WORKSPACE and
 *              enqueues nothing
 *   set-up     the first call on a device looks up the array's device address
 *              (cudaGetSymbolAddress) with that device current; make that first
 *              call before any stream capture.  The address is kept for the
 *              life of the process: after a cudaDeviceReset it is stale, so a
 *              process that resets a device must not call this entry point on
 *              that device again
 *   sharing    every call on a device uses the same array, which keeps the last
 *              call's descriptors; each call rewrites every descriptor its
 *              kernel reads before the kernel runs, so nothing needs clearing,
 *              but calls that overlap on the GPU (different streams, no ordering
 *              between them) race on the array and must be serialised
 * It calls no cudaMalloc or cudaFree and uses no heap memory on the host.
 */
int nf4_backward_a_batched_noalloc(const nf4_problem* problems, int count, void* stream);

/*
 * Dense weight gradient of a matrix product C = A @ B:
 *
 *     grad_B[K x N] = A[M x K]^T @ grad_C[M x N]
 *
 * (page "trueno-gpu 0.4.17 -- src/kernels/backward/mod.rs": the backward
 * module's GEMM kernels give the gradients of both operands of a matrix
 * product; GemmBackwardBKernel takes a_ptr and writes grad_b_ptr.  The page
 * does not print that kernel; this is the plain definition.)  Beside a frozen
 * NF4 base weight it is the gradient of the trainable 16-bit weights (LoRA
 * adapters or fully trained layers): the sum runs over the M tokens, both
 * operands are 16-bit floats of one type, products are summed in fp32 by the
 * tensor cores (tcgen05 pair MMAs, both operands loaded by TMA as they are).
 *   A, grad_C  [M][K] and [M][N], row-major, NF4_BF16 or NF4_F16 (`dtype`,
 *              both), 16-byte aligned; K and N positive multiples of 8
 *   grad_B     [K][N] fp32, 16-byte aligned, overwritten; M == 0 writes zeros
 *   workspace  when the output tiles are too few to occupy the GPU, the tokens
 *              are cut into nf4_gemm_backward_b_splits(M, K, N, pairs) runs
 *              whose fp32 partial sums go to the workspace and are added in
 *              run order by a second kernel (deterministic);
 *              nf4_gemm_backward_b_ws_bytes(M, K, N) bytes (0: none needed),
 *              256-byte aligned; with less (or NULL) the call splits less (or
 *              not at all) and gives the same values up to fp32 summation order
 * Returns NF4_ERR_INVALID or NF4_ERR_ALIGN (nothing enqueued) for arguments
 * outside these rules.
 */
int nf4_gemm_backward_b_splits(int M, int K, int N, int pairs);
size_t nf4_gemm_backward_b_ws_bytes(int M, int K, int N);
int nf4_gemm_backward_b(const void* A, const void* grad_C, int dtype, float* grad_B, int M, int K,
                        int N, void* workspace, size_t workspace_bytes, void* stream);

/*
 * Synchronise `stream`, then report and clear the library's device status word
 * (NF4_ERR_TIMEOUT if any kernel's bounded wait gave up since the last check),
 * or NF4_ERR_CUDA if the stream reports a CUDA error.
 */
int nf4_check_error(void* stream);

/*
 * As nf4_check_error, and if a wait gave up, where the first one was: site[0] =
 * block index + 1, site[1] = thread index, site[2] = the shared-memory address
 * waited on, site[3] = the phase parity or flag value it waited for.  `site`
 * (4 words, host memory) is zeroed when there was no timeout; may be NULL.
 */
int nf4_check_error_site(void* stream, unsigned int* site);

/*
 * Self-test of the bounded waits that every kernel of this library uses (no
 * counterpart on the pages).  Enqueues on `stream` one CTA whose waits can never
 * be satisfied: one thread waits on an mbarrier that nothing arrives on, with a
 * limit of limit_cycles SM clock cycles, gives up, records NF4_ERR_TIMEOUT and
 * where it waited in the library's status word (the same path a stalled
 * pipeline takes), and raises the CTA's abort flag; a second thread, waiting
 * with the normal limit on another such barrier, must return as soon as it
 * sees that flag.  Both exit; the GPU context stays usable.  The next
 * nf4_check_error_site then reports NF4_ERR_TIMEOUT with site = {1 (block 0),
 * 0 (thread 0), the barrier's shared-memory address, 0 (parity)} and clears it.
 *   limit_cycles  1000 .. 2e9
 *   where         device memory for 3 words: [0] the barrier's shared-memory
 *                 address, [1] 1 if the first wait returned success (it must
 *                 not), [2] 1 if the second wait did (it must not)
 * Returns NF4_ERR_INVALID for arguments outside these rules (nothing enqueued).
 */
int nf4_watchdog_selftest(long long limit_cycles, unsigned int* where, void* stream);

/*
 * Backward of RMS layer normalisation (page "trueno-gpu 0.4.17 --
 * src/kernels/backward/rms_norm.rs", module doc: forward y_i = x_i * gamma_i /
 * r per row, r = sqrt(mean(x^2) + eps) kept by the forward pass; the kernel's
 * parameters input, gamma, rms, grad_output, grad_input, num_rows,
 * hidden_dim).  Computes the gradient of that forward:
 *   grad_input[row][i] = gamma_i * g_i / r - x_i * mean_j(x_j g_j gamma_j) / r^3
 *   grad_gamma[i]      = sum over rows of g_i * x_i / r        (if grad_gamma != NULL)
 * with g = grad_output.  The page's kernel multiplies the second term of
 * grad_input by gamma_i too and adds eps to r^2 again; neither is done here
 * (the page's own test criterion, agreement with finite differences, rules
 * them out), and eps is not needed since r holds it.  Rows need not fit a warp.
 *   input, grad_output, grad_input  [num_rows][hidden_dim] fp32, 16-byte aligned
 *   gamma [hidden_dim] fp32, 16-byte aligned; rms [num_rows] fp32, 4-byte aligned
 *   hidden_dim  multiple of 4, at most 8192; num_rows >= 0 (0: grad_gamma zeroed)
 *   workspace   with grad_gamma: caller-owned device memory, 16-byte aligned, at
 *               least rms_norm_backward_ws_bytes(num_rows, hidden_dim) bytes
 *               (per-CTA partial sums, summed in CTA order: deterministic)
 * Returns NF4_ERR_INVALID, NF4_ERR_ALIGN or NF4_ERR_WORKSPACE (nothing
 * enqueued) for arguments outside these rules.
 */
size_t rms_norm_backward_ws_bytes(int num_rows, int hidden_dim);
int rms_norm_backward(const float* input, const float* gamma, const float* rms,
                      const float* grad_output, float* grad_input, float* grad_gamma,
                      int num_rows, int hidden_dim, void* workspace, size_t workspace_bytes,
                      void* stream);

#ifdef __cplusplus
}
#endif
#endif /* NF4BWD_H */
