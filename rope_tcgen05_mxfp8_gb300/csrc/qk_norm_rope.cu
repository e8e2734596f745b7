// Kernel K2: the norm/RoPE work on the Q/K hand-off as a kernel of its own (the
// method and the task layout are described in qk_norm_rope.cuh); the default. With
// QKV_CTE_FLAG_NORM_IN_GEMM the CTA-pair GEMM's epilogue warps do this work between
// tiles instead.
//
// Launched as a programmatic dependent of K1, its blocks run beside K1's persistent
// CTAs and take each task once K1's counter says the task's 128-row panel is complete
// (a bounded acquire wait), so it mostly hides under the GEMM. Alone (serial flag) it
// is an HBM-bound pass over the hand-off.
//
// Beside K1, warps claim tasks in order from a counter. A warp that shares its SM
// sub-partition with the TMA-load or MMA-issue warp of the K1 CTA on its SM (K1
// publishes them per SM) holds back until that CTA has finished, or until every GEMM
// pair has reached the claimed tail of its tile sequence (the GEMM then balances the
// pairs itself, and the pass must not be left with a backlog when it ends), then joins
// for the tasks left: sharing those schedulers slows the GEMM about twice as much per
// unit of this work as running on the other two sub-partitions. The per-head norms' tasks are
// heavier (the statistics of every head): with fewer warps they would fall behind the
// GEMM, so there, as when the pass runs alone, every warp takes every gridDim-th task
// (no counter on the critical path).
#include "qk_norm_rope.cuh"

namespace qkvcte {

namespace {

constexpr int kThreads = 128;
// Heads per warp task: at most 20 (small tasks keep the warps evenly loaded to the
// end); fewer when the problem is small, so that every warp of the grid gets a task
// (the 512-token cross-attention K|V call: 4 heads per task, 640 tasks for 608 warps
// instead of 128 tasks of 20 heads, which ran latency-bound on 32 blocks).
constexpr int kHeadGroups[] = {20, 10, 5, 4, 2, 1};

int head_group_for(const NormRopeArgs& a, long long warps) {
  for (int g : kHeadGroups)
    if (nrp::task_count(a, g) >= warps) return g;
  return 1;
}

// Lane 0: hold back (bounded) while the K1 CTA on this SM occupies this warp's
// sub-partition with its load or MMA warp and tasks remain.
__device__ __forceinline__ void defer_while_busy(const NormRopeArgs& p, long long tasks) {
  if (p.sm_busy == nullptr) return;
  const uint32_t* busy = p.sm_busy + (nrp::sm_id() & (kSmTable - 1));
  const uint32_t bit = 1u << (nrp::warp_slot() & 3);
  if (!(nrp::ld_relaxed(busy) & bit)) return;
  const unsigned long long t0 = nrp::now_ns();
  while (true) {
    __nanosleep(2000);
    if (!(nrp::ld_relaxed(busy) & bit)) return;
    if (static_cast<long long>(nrp::ld_relaxed(p.task_next)) >= tasks) return;
    if (p.gemm_claims != nullptr && nrp::ld_relaxed(p.gemm_claims) >= p.release_at) return;
    if (nrp::now_ns() - t0 > nrp::kWaitLimitNs) return;  // a hint only: go ahead
  }
}

// kBatch: heads whose hand-off loads a lane keeps in flight. Beside the GEMM (one block
// per SM fits there) 4; alone, the across-heads form takes 2: 168 registers instead of
// 240 let three blocks share an SM instead of two, and more warps hide more latency
// than deeper batches (measured at 480p: 0.260 against 0.2875 ms alone, 5.37 TB/s;
// beside the GEMM 2 was no better).
template <bool kHeadStats, int kBatch>
__global__ void __launch_bounds__(kThreads) qk_norm_rope_kernel(const __grid_constant__ NormRopeArgs p) {
  if (threadIdx.x == 0) atomicMin(&p.stamps[0], nrp::now_ns());
  const int lane = threadIdx.x & 31;
  const long long tasks = nrp::task_count(p, p.head_group);
  if (p.claim && lane == 0) defer_while_busy(p, tasks);
  __syncwarp();
  // Read-once hand-off and write-once output: first out of L2, so the GEMM's
  // L2-resident weight band running beside this pass keeps its place.
  const uint64_t once = nrp::evict_first_policy();
  const long long warps = static_cast<long long>(gridDim.x) * (kThreads / 32);
  long long task = static_cast<long long>(blockIdx.x) * (kThreads / 32) + (threadIdx.x >> 5) - warps;
  while (true) {
    int ok = 1;
    if (lane == 0) {
      task = p.claim ? static_cast<long long>(atomicAdd(p.task_next, 1u)) : task + warps;
      if (task < tasks) ok = nrp::wait_panel_ready(p.ready + nrp::task_panel(p, task, p.head_group), p.ready_target);
    }
    task = __shfl_sync(0xffffffffu, task, 0);
    if (task >= tasks) break;
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (!ok) {
      if (lane == 0) atomicOr(p.status, kErrNormReadyWait);
      break;
    }
    nrp::run_task<kHeadStats, kBatch>(p, task, p.head_group, once);
  }
  if (threadIdx.x == 0) atomicMax(&p.stamps[1], nrp::now_ns());
}

}  // namespace

cudaError_t launch_norm_rope(const NormRopeArgs& a, cudaStream_t s, int num_sms, bool overlap) {
  if (!a.norm && !a.rope) return cudaSuccess;
  if (a.d_head < 32 || a.d_head % 32 != 0) return cudaErrorInvalidValue;
  if (nrp::task_count(a, kHeadGroups[0]) == 0) return cudaSuccess;
  // Overlapped with the GEMM, the grid is kept to what fits beside each GEMM CTA
  // (registers are the limit) so every block finds its tasks as their panels
  // complete. That sizing only affects speed: the GEMM never waits for this kernel.
  // Alone, the pass takes every SM it can hold.
  const auto kernel = a.head_kind != 0 ? qk_norm_rope_kernel<true, nrp::kHeadBatch>
                      : overlap        ? qk_norm_rope_kernel<false, nrp::kHeadBatch>
                                       : qk_norm_rope_kernel<false, 2>;
  int per_sm = 1;
  if (!overlap) {
    int occ = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kernel, kThreads, 0) == cudaSuccess && occ > per_sm)
      per_sm = occ;
  }
  NormRopeArgs args = a;
  args.head_group = head_group_for(a, static_cast<long long>(per_sm) * num_sms * (kThreads / 32));
  const long long tasks = nrp::task_count(a, args.head_group);
  long long blocks = (tasks + kThreads / 32 - 1) / (kThreads / 32);
  if (blocks > static_cast<long long>(per_sm) * num_sms) blocks = static_cast<long long>(per_sm) * num_sms;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(blocks));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = overlap ? 1 : 0;
  args.claim = overlap && a.head_kind == 0 ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, args);
}

}  // namespace qkvcte
