// nf4_trace.cuh -- optional timing probes, compiled in only with -DNF4_TRACE.
//
// The first CTAs of a launch record clock64() at fixed points of each role
// into a device buffer [cta][event][slot] set with nf4_debug_set_trace(); the
// event numbers are listed at each kernel.  Without NF4_TRACE the probes expand
// to nothing.
#pragma once

namespace nf4 {
// Pair kernel (bwd_a_kernel):
// the CTAs of clusters 0 and 1 record clock64() at fixed points of each role into
// a device buffer [cta][event][slot]; event kTraceEvents-1 slot 0 is the clock
// right after the start-up cluster barrier, the common reference of both CTAs.
// Events: 0-15 converter warp after its operand-slot wait, 16-31 converter warp
// done, 32/33/38 MMA before wait / after wait / after commit, 35/36 epilogue
// tile start / end, 39 reference, 40 producer issue, 41 watcher sees stage,
// 42 converter group leader sees raw data, 43 converter group leader starts,
// 44 slot 0 kernel entry / slot 1 all roles done / slot 2 after the last
// cluster barrier; pre-converted variant: 45 A producer issues the stage's A
// copy, 46 watcher sees both A copies landed; epilogue: 34 slot k = item k's
// partial sums written and counted, 37 slot k = item k's partner counts all
// seen; 48-63 converter warp 0-15 has
// stored its B^T chunks, 64-79 it has also passed the proxy fence; epilogue
// warp 0, a pair's last item (slot 16 * M-block + chunk): 83 chunk loaded from
// TMEM, 80 chunk staged, 81 (slot M-block) proxy fence passed, 82 stores
// issued; 84 slot 0: the epilogue's stores have completed.
//
// Few-token kernel (small_m_kernel), CTAs 0 and 1 (k-tile 0, cluster ranks 0
// and 1 when S > 1): slot s of events 0-6 and 8 is stage s.  0 producer issues
// the NF4 box, 1 producer issues grad_out box 0, 2 first warp of the group has
// the raw stage, 3 it has the operand slot, 4 it has finished the stage, 8 the
// group's last warp has finished it, 5 MMA thread has the stage, 6 MMA thread
// has committed it.  Event 7: slot 0 after start-up (the reference), 1
// accumulator ready, 2 partial tile written, 3 after the first cluster
// barrier, 4 reduction stored, 5 after the last cluster barrier.
#ifdef NF4_TRACE
__device__ unsigned long long* g_trace = nullptr;
constexpr int kTraceSlots = 512;
constexpr int kTraceEvents = 88;
constexpr unsigned kTraceCtas = 4;  // the first two pairs
// Each kernel caches the buffer pointer once (NF4_TRACE_INIT), so a probe is a
// clock read and one store.
#define NF4_TRACE_INIT unsigned long long* const nf4_trace_buf = blockIdx.x < kTraceCtas ? g_trace : nullptr
#define NF4_PROBE(ev, idx)                                                               \
  do {                                                                                   \
    if (nf4_trace_buf != nullptr && (idx) < kTraceSlots)                                 \
      nf4_trace_buf[(blockIdx.x * kTraceEvents + (ev)) * kTraceSlots + (idx)] =           \
          static_cast<unsigned long long>(clock64());                                    \
  } while (0)
#else
#define NF4_TRACE_INIT do { } while (0)
#define NF4_PROBE(ev, idx) do { } while (0)
#endif

// Progress counters (compiled in only with -DNF4_PROGRESS, for diagnosing a
// stall): each role of each CTA stores how far it got into
// g_progress[block][slot]; slots are listed at the kernel.
#ifdef NF4_PROGRESS
__device__ unsigned int* g_progress = nullptr;
#define NF4_PROGRESS_SET(slot, value)                                                   \
  do {                                                                                 \
    if (g_progress != nullptr)                                                         \
      *reinterpret_cast<volatile unsigned int*>(g_progress + blockIdx.x * 32 + (slot)) = \
          static_cast<unsigned int>(value);                                            \
  } while (0)
#else
#define NF4_PROGRESS_SET(slot, value) do { } while (0)
#endif

}  // namespace nf4
